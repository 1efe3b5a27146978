"""Device twin of the generator: fills torch CUDA tensors with the same bytes
that ``synth`` produces on the CPU (for weight sets too large to draw on the
host).  Input plumbing only; holds none of the layer's arithmetic."""
from __future__ import annotations

import ctypes
import os

import torch

from . import (LayerShape, SIGMA_Z, WEIGHT_STD, expert_matrix_key, make_key)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = os.path.join(_HERE, "libcolisynth.so")
        if not os.path.exists(path):
            from .build import build
            build()
        lib = ctypes.CDLL(path)
        lib.synth_quant_rows.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_quant_groups64.argtypes = lib.synth_quant_rows.argtypes
        lib.synth_normal_f32.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_longlong,
                                         ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
        _LIB = lib
    return _LIB


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def fill_expert_records(shape: LayerShape, seed, layer, kind, experts, out: torch.Tensor,
                        scales: torch.Tensor, first_slot: int = 0):
    """Write the records of ``experts`` (ids) into ``out`` [n, record_bytes]
    uint8 and ``scales`` [n, scale_count] f32, starting at row ``first_slot``."""
    lib = _lib()
    inter = shape.inter if kind == "routed" else shape.shared_inter
    H = shape.hidden
    qmax = shape.qmax
    c = WEIGHT_STD / (SIGMA_Z * qmax)
    rbH = shape.row_bytes(H)
    rbI = shape.row_bytes(inter)
    offs = [0, inter * rbH, 2 * inter * rbH]
    dims = [(inter, H), (inter, H), (H, inter)]
    gs = shape.group_size
    if gs not in (0, 64):
        raise ValueError("the device generator draws per-row or 64-element groups")
    per = [r if not gs else r * k // gs for r, k in dims]
    soffs = [0, per[0], per[0] + per[1]]
    fn = lib.synth_quant_groups64 if gs else lib.synth_quant_rows
    for n, e in enumerate(experts):
        row = first_slot + n
        base = out[row].data_ptr()
        sbase = scales[row].data_ptr()
        for m in range(3):
            k0, k1 = expert_matrix_key(seed, layer, kind, int(e), m)
            rows, K = dims[m]
            rc = fn(k0, k1, rows, K, qmax, c, shape.weight_bits,
                                      ctypes.c_void_p(base + offs[m]),
                                      ctypes.c_void_p(sbase + 4 * soffs[m]), _stream())
            if rc:
                raise RuntimeError(f"synth_quant_rows failed ({rc})")
    del rbI


def expert_records(shape: LayerShape, seed, layer, kind, n, device="cuda"):
    inter = shape.inter if kind == "routed" else shape.shared_inter
    out = torch.empty((n, shape.record_bytes(inter)), dtype=torch.uint8, device=device)
    sc = torch.empty((n, shape.scale_count(inter)), dtype=torch.float32, device=device)
    fill_expert_records(shape, seed, layer, kind, range(n), out, sc)
    return out, sc


def normal_f32(key, n, std, device="cuda"):
    out = torch.empty(n, dtype=torch.float32, device=device)
    mul = float(torch.tensor(std / SIGMA_Z, dtype=torch.float32))
    rc = _lib().synth_normal_f32(key[0], key[1], n, mul, ctypes.c_void_p(out.data_ptr()), _stream())
    if rc:
        raise RuntimeError("synth_normal_f32 failed")
    return out


def token_batch(shape: LayerShape, seed, stream, positions, device="cuda"):
    """Rows x ~ N(0,1) for (stream, position, attempt 0), drawn on the device."""
    rows = [normal_f32(make_key(seed, "x", stream, int(p), 0), shape.hidden, 1.0, device)
            for p in positions]
    return torch.stack(rows) if rows else torch.empty((0, shape.hidden), device=device)
