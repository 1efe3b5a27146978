"""The C-ABI library loads and exports every function include/*.h declares
(no GPU needed; no compute calls)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "quantized_expert_ffn_sigmoid_gb300", "libcolimoe.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(coli_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("coli_moe_route", "coli_moe_quantize_act", "coli_moe_forward"):
        assert required in names
    assert len(names) >= 11


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_exports_match_header():
    import quantized_expert_ffn_sigmoid_gb300 as cm
    assert sorted(cm.EXPORTS) == declared_functions()
    for name in cm.EXPORTS:
        assert callable(getattr(cm, name))


def test_host_only_entry_points(lib):
    # pure host logic: sizes, layouts and messages need no GPU
    import synth
    import quantized_expert_ffn_sigmoid_gb300 as cm
    cfg = cm.Cfg.of(synth.GLM)
    n1 = cm.coli_moe_workspace_size(cfg, 1)
    n2048 = cm.coli_moe_workspace_size(cfg, 2048)
    assert 0 < n1 < n2048
    L = cm.coli_moe_workspace_layout(cfg, 4)
    assert L.total == cm.coli_moe_workspace_size(cfg, 4)
    offs = [L.status, L.n_entries, L.entry_expert, L.qx, L.dx, L.qh, L.dh, L.o]
    assert all(o % 16 == 0 for o in offs) and L.o < L.total
    assert cm.coli_moe_strerror(cm.COLI_EWORKSPACE) == "workspace too small"
    # the header cleared by coli_moe_workspace_init (status block, device
    # counters, router exchange words) is the size the header file states,
    # and the tables start after it
    import re
    doc = open(os.path.join(ROOT, "include", "coli_moe.h")).read()
    cleared = int(re.search(r"min\(ws_bytes, (\d+)\) bytes", doc).group(1))
    assert L.status == 0 and cleared <= L.n_entries
    bad = cm.Cfg.of(synth.GLM)
    bad.hidden = 100
    assert cm.coli_moe_workspace_size(bad, 4) == 0
    bad = cm.Cfg.of(synth.GLM)
    bad.top_k = 40
    assert cm.coli_moe_workspace_size(bad, 4) == 0


def test_group_size_host_checks(lib):
    # group scales: 0 (per row) or 64, and only with int4 codes
    import dataclasses
    import synth
    import quantized_expert_ffn_sigmoid_gb300 as cm
    gs = cm.Cfg.of(synth.GLM_GS64)
    assert gs.group_size == 64
    assert cm.coli_moe_workspace_size(gs, 4) == cm.coli_moe_workspace_size(cm.Cfg.of(synth.GLM), 4) > 0
    for bad in (dataclasses.replace(synth.GLM_GS64, group_size=32),
                dataclasses.replace(synth.GLM_GS64, weight_bits=8)):
        assert cm.coli_moe_workspace_size(cm.Cfg.of(bad), 4) == 0
    assert cm.Cfg.of(synth.GLM).group_size == 0


def test_weight_bits_host_checks(lib):
    # 2, 4 or 8 bits; group scales only with int4 (not with packed int2)
    import dataclasses
    import synth
    import quantized_expert_ffn_sigmoid_gb300 as cm
    n4 = cm.coli_moe_workspace_size(cm.Cfg.of(synth.GLM), 4)
    assert cm.coli_moe_workspace_size(cm.Cfg.of(synth.GLM_INT2), 4) == n4 > 0
    assert cm.coli_moe_workspace_size(cm.Cfg.of(synth.TINY_INT2), 4) > 0
    for bad in (dataclasses.replace(synth.GLM_INT2, group_size=64),
                dataclasses.replace(synth.GLM, weight_bits=3),
                dataclasses.replace(synth.GLM, weight_bits=1)):
        assert cm.coli_moe_workspace_size(cm.Cfg.of(bad), 4) == 0


def test_expert_parallel_host_checks(lib):
    # shard 0 holds the shared experts' pairs, the other shards do not; the
    # shard index must lie in [0, ep_size), ep_size in [0, n_experts]
    import synth
    import quantized_expert_ffn_sigmoid_gb300 as cm
    whole = cm.coli_moe_workspace_size(cm.Cfg.of(synth.GLM), 32)
    assert cm.coli_moe_workspace_size(cm.Cfg.of(synth.GLM, 0, 1), 32) == whole
    assert cm.coli_moe_workspace_size(cm.Cfg.of(synth.GLM, 0, 4), 32) == whole
    assert 0 < cm.coli_moe_workspace_size(cm.Cfg.of(synth.GLM, 3, 4), 32) < whole
    for rank, size in ((4, 4), (-1, 2), (1, 1), (1, 0), (0, 257), (0, -2)):
        assert cm.coli_moe_workspace_size(cm.Cfg.of(synth.GLM, rank, size), 32) == 0, (rank, size)
