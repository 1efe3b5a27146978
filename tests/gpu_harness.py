"""GPU-side harness for the parity tests: builds a layer on the device, runs
the library through its C ABI and compares every observable with the oracle.
Imported only by tests marked ``gpu``."""
from __future__ import annotations

import concurrent.futures as cf
import os
import threading

import numpy as np
import torch

import oracle
import synth
import quantized_expert_ffn_sigmoid_gb300 as cm
from helpers import elementwise_err, normwise_err, unpermute_int2, unpermute_int4

Y_TOL = 1e-3     # max normwise relative error of the layer output
W_RTOL = 1e-5    # gate weights: fp32 router vs fp64 oracle


class DeviceLayer:
    """One MoE layer's weights on the GPU plus lazily copied host views."""

    def __init__(self, shape, seed, layer=0, device_weights=False, bias="uniform", dev="cuda"):
        self.shape, self.seed, self.layer, self.dev = shape, seed, layer, dev
        self.cfg = cm.Cfg.of(shape)
        if device_weights:
            import synth.gpu as sg
            self.recs, self.scs = sg.expert_records(shape, seed, layer, "routed", shape.n_experts, dev)
            if shape.n_shared:
                self.srec, self.ssc = sg.expert_records(shape, seed, layer, "shared", shape.n_shared, dev)
            else:
                self.srec = self.ssc = None
            self._host = {}
        else:
            routed = [synth.expert_record(shape, seed, layer, "routed", e) for e in range(shape.n_experts)]
            shared = [synth.expert_record(shape, seed, layer, "shared", s) for s in range(shape.n_shared)]
            self._host = {("routed", e): r for e, r in enumerate(routed)}
            self._host.update({("shared", s): r for s, r in enumerate(shared)})
            t = lambda a: torch.from_numpy(np.ascontiguousarray(np.stack(a))).to(dev)
            self.recs, self.scs = t([r for r, _ in routed]), t([s for _, s in routed])
            if shared:
                self.srec, self.ssc = t([r for r, _ in shared]), t([s for _, s in shared])
            else:
                self.srec = self.ssc = None
        self.W = cm.make_weights(self.recs, self.scs, self.srec, self.ssc)
        self.router_w = synth.router_weight(shape, seed, layer)
        self.bias = {"uniform": lambda: synth.router_bias(shape, seed, layer),
                     "zipf": lambda: synth.zipf_router_bias(shape, seed, layer),
                     "zero": lambda: synth.zero_router_bias(shape)}[bias]()
        self.wr_d = torch.from_numpy(self.router_w).to(dev)
        self.bias_d = torch.from_numpy(self.bias).to(dev)

    def get_record(self, kind, e):
        key = (kind, int(e))
        if key not in self._host:
            if kind == "routed":
                self._host[key] = (self.recs[e].cpu().numpy(), self.scs[e].cpu().numpy())
            else:
                self._host[key] = (self.srec[e].cpu().numpy(), self.ssc[e].cpu().numpy())
        return self._host[key]

    # ------------------------------------------------------------------ runs
    def run(self, x: np.ndarray, dump=True, ws=None, route=True, idx=None, w=None, layer=False, cfg=None,
            W=None, shape=None):
        """Route (unless idx/w given) and forward; returns the GPU observables.
        ``layer``: one coli_moe_layer call (router and experts together).
        ``cfg`` / ``W`` / ``shape``: another config and weights of this
        layer (e.g. one shard of an expert-parallel layer)."""
        shape, dev = shape or self.shape, self.dev
        cfg_ = self.cfg if cfg is None else cfg
        W_ = self.W if W is None else W
        T, k = x.shape[0], shape.top_k
        xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)
        if ws is None:
            ws = cm.new_workspace(cfg_, T)
        if layer:
            idx_d = torch.full((T, k), -7, dtype=torch.int32, device=dev)
            w_d = torch.full((T, k), -7.0, dtype=torch.float32, device=dev)
            dump = False
        elif route:
            idx_d = torch.full((T, k), -7, dtype=torch.int32, device=dev)
            w_d = torch.full((T, k), -7.0, dtype=torch.float32, device=dev)
            cm.coli_moe_route(cfg_, xd, self.wr_d, self.bias_d, idx_d, w_d, ws)
        else:
            idx_d = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(dev)
            w_d = torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(dev)
        y = torch.full((T, shape.hidden), float("nan"), dtype=torch.float32, device=dev)
        L = cm.coli_moe_workspace_layout(cfg_, T)
        P = T * k + shape.n_shared * T
        imax = max(shape.inter, shape.shared_inter if shape.n_shared else 0)
        acc_gu = acc_d = None
        if layer:
            cm.coli_moe_layer(cfg_, W_, xd, self.wr_d, self.bias_d, idx_d, w_d, y, ws)
        elif dump:
            acc_gu = torch.zeros((P, 2, imax, shape.hidden // 32), dtype=torch.int32, device=dev)
            acc_d = torch.zeros((P, shape.hidden, imax // 32), dtype=torch.int32, device=dev)
            cm.coli_moe_forward_dump(cfg_, W_, xd, idx_d, w_d, y, ws, acc_gu, acc_d)
        else:
            cm.coli_moe_forward(cfg_, W_, xd, idx_d, w_d, y, ws)
        status = cm.coli_moe_status(ws)
        wsh = ws.cpu().numpy()

        def view(off, dtype, count):
            return np.frombuffer(wsh[off:off + np.dtype(dtype).itemsize * count].tobytes(), dtype)

        n_ent = int(view(L.n_entries, np.int32, 1)[0])
        out = dict(idx=idx_d.cpu().numpy(), w=w_d.cpu().numpy(), y=y.cpu().numpy(), status=status,
                   n_entries=n_ent,
                   entry_expert=view(L.entry_expert, np.int32, n_ent),
                   entry_count=view(L.entry_count, np.int32, n_ent),
                   entry_offset=view(L.entry_offset, np.int32, n_ent + 1),
                   pair_token=view(L.pair_token, np.int32, P),
                   slot=view(L.pair_slot_of, np.int32, T * k).reshape(T, k))
        qx = view(L.qx, np.int8, T * shape.hidden).reshape(T, shape.hidden)
        qh = view(L.qh, np.int8, P * imax).reshape(P, imax)
        if shape.weight_bits == 4:
            qx, qh = unpermute_int4(qx), unpermute_int4(qh)
        elif shape.weight_bits == 2:
            qx, qh = unpermute_int2(qx), unpermute_int2(qh)
        out.update(qx=qx, dx=view(L.dx, np.float32, T * shape.hidden // 32).reshape(T, -1),
                   qh=qh, dh=view(L.dh, np.float32, P * imax // 32).reshape(P, -1))
        if dump:
            out.update(acc_gu=acc_gu.cpu().numpy(), acc_d=acc_d.cpu().numpy())
        return out


def _pool_size():
    return max(1, min(16, os.cpu_count() or 1))


def check_parity(layer: DeviceLayer, x, g, ref=None, idx=None, w=None, tokens=None, threads=None,
                 max_tokens=32):
    """Compare GPU observables ``g`` with the oracle.  ``tokens`` restricts the
    expert-level comparisons (and y) to a sample of positions.

    The oracle evaluates the sampled positions expert by expert, in runs of at
    most ``max_tokens`` positions on a thread pool (evaluation order only); each
    run's pairs are compared as they come, so full-size layers are checked in
    bounded memory."""
    shape = layer.shape
    T = x.shape[0]
    H = shape.hidden
    assert g["status"] == 0, f"device status {g['status']}"
    if idx is None:
        logits = oracle.router_logits(x, layer.router_w)
        ridx, rw = oracle.route(logits, layer.bias, shape)
        assert np.array_equal(g["idx"], ridx), "routing indices differ"
        np.testing.assert_allclose(g["w"], rw, rtol=W_RTOL, atol=1e-7)
        idx, w = ridx, rw            # the oracle runs on its own routing
    tabs = oracle.union_tables(idx, shape.n_experts, shape.n_shared)
    n_ent = tabs["counts"].size
    assert g["n_entries"] == n_ent
    exp_ids = np.concatenate([tabs["uniq"], shape.n_experts + np.arange(shape.n_shared)])
    assert np.array_equal(g["entry_expert"], exp_ids)
    assert np.array_equal(g["entry_count"], tabs["counts"])
    assert np.array_equal(g["entry_offset"], tabs["offsets"])
    npair = int(tabs["offsets"][-1])
    assert np.array_equal(g["pair_token"][:npair], tabs["pair_token"])
    assert np.array_equal(g["slot"], tabs["slot"])
    qx, dx = oracle.q8_0_quantize(x.astype(np.float32))
    assert np.array_equal(g["qx"], qx), "Q8_0 codes of x differ"
    assert np.array_equal(g["dx"], dx), "Q8_0 scales of x differ"

    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    w = np.asarray(w, np.float64)
    # host copies of the records the sampled positions use, fetched up front
    for e in np.unique(idx[sel][(idx[sel] >= 0) & (idx[sel] < shape.n_experts)]):
        layer.get_record("routed", int(e))
    for s in range(shape.n_shared):
        layer.get_record("shared", s)

    lock = threading.Lock()
    stats = dict(qh_checked=0, qh_unstable=0, qh_flips=0, accd_blocks=0, pairs=0)
    y_delta = np.zeros((sel.size, H))   # linear effect of the GPU's admissible qh steps
    bound = np.zeros((sel.size, H))     # elementwise bound on |y_gpu - y_oracle|
    stepped = np.zeros(sel.size, bool)  # positions with an admissible qh step in any of their pairs
    gsz = shape.group_size

    def on_entry(kind, e, pr):
        inter = shape.inter if kind == "routed" else shape.shared_inter
        tl = pr["tokens"]                      # indices into sel
        ts = sel[tl]
        if kind == "routed":
            ps = g["slot"][ts, pr["js"]].astype(np.int64)
            wt = w[ts, pr["js"]]
        else:
            ps = int(tabs["offsets"][tabs["uniq"].size + e]) + ts
            wt = np.ones(ts.size)
        if "acc_gu" in g:
            assert np.array_equal(g["acc_gu"][ps, 0, :inter], pr["acc_g"]), "gate block dots differ"
            assert np.array_equal(g["acc_gu"][ps, 1, :inter], pr["acc_u"]), "up block dots differ"
        qh_g = g["qh"][ps, :inter].astype(np.int64)
        qh_r = pr["qh"].astype(np.int64)
        st = pr["qh_stable"]
        assert np.array_equal(qh_g[st], qh_r[st]), "requantised h differs where unique"
        assert np.abs(qh_g - qh_r).max(initial=0) <= 1
        # block scale: amax/127 of h, within the h error bound of the oracle
        nb = inter // 32
        dh = pr["dh"].astype(np.float64)                                          # [n, nb]
        ddh = 4.0 * pr["h_err"].reshape(-1, nb, 32).max(axis=2) / 127.0 + np.abs(dh) * 2.0 ** -21
        assert np.all(np.abs(g["dh"][ps, :nb].astype(np.float64) - dh) <= ddh), "dh outside its bound"
        blk_ok = (qh_g == qh_r).reshape(-1, nb, 32).all(axis=2)                    # [n, nb]
        if "acc_d" in g:
            # bit-exact given the same codes: every block whose 32 h codes the
            # GPU and the oracle agree on (all of them unless a non-unique
            # code took its other admissible value)
            ad = g["acc_d"][ps, :, :nb]                                           # [n, H, nb]
            ok = np.broadcast_to(blk_ok[:, None, :], ad.shape)
            assert np.array_equal(ad[ok], pr["acc_d"][ok]), "down block dots differ"
        # Where the GPU took the other admissible code of a non-unique h
        # value (asserted above: |dq| <= 1 and only there), the oracle's
        # output for the GPU's codes is the oracle's own plus the linear
        # effect of those steps on the down product.  The elementwise bound
        # covers the unadjusted difference: fp32 evaluation plus the effect
        # of every +-1 step.
        rec, sc = layer.get_record(kind, e)
        wd = oracle.unpack_weight_rows(np.asarray(rec).reshape(-1)[2 * inter * shape.row_bytes(H):],
                                       H, inter, shape.weight_bits).astype(np.float64)
        sc = np.asarray(sc, np.float64)
        if gsz:  # the down matrix's scales: [H][inter/g] after gate and up
            s_blk = np.repeat(sc[2 * inter * H // gsz:].reshape(H, inter // gsz), gsz // 32, axis=1)
        else:
            s_blk = np.repeat(sc[2 * inter:2 * inter + H][:, None], nb, axis=1)
        wd_s = wd * np.repeat(s_blk, 32, axis=1)                                  # dequantised down weights
        dqs = (qh_g - qh_r).astype(np.float64)                                     # [n, inter]
        adj = (wd_s @ (dqs * np.repeat(dh, 32, axis=1)).T).T                       # [n, H]
        flip = (np.abs(wd_s) @ (np.abs(dqs) * np.repeat(dh + ddh, 32, axis=1)).T).T
        acc_term = np.einsum("hb,nhb,nb->nh", np.abs(s_blk), np.abs(pr["acc_d"]).astype(np.float64), ddh)
        term = 4.0 * pr["o_err"] + acc_term + flip
        # combine rounding (fp32, k + n_shared terms) and fp32 gate weights
        bnd = np.abs(wt)[:, None] * (term + np.abs(pr["o"]) * (2.0 ** -20 + 2e-6))
        with lock:
            stepped[tl[(qh_g != qh_r).any(axis=1)]] = True
            np.add.at(y_delta, tl, wt[:, None] * adj)
            np.add.at(bound, tl, bnd)
            stats["qh_checked"] += qh_g.size
            stats["qh_unstable"] += int((~st).sum())
            stats["qh_flips"] += int((qh_g != qh_r).sum())
            stats["accd_blocks"] += int(blk_ok.sum()) * H
            stats["pairs"] += tl.size

    n_thr = threads or (_pool_size() if sel.size * shape.hidden > 65536 else 1)
    with cf.ThreadPoolExecutor(n_thr) as ex:
        ref = oracle.moe_forward(shape, layer.get_record, x[sel], idx[sel], w[sel], on_entry=on_entry,
                                 map_fn=ex.map, max_tokens=max_tokens)
    y_g = g["y"][sel]
    err = normwise_err(y_g, ref["y"] + y_delta)
    assert err <= Y_TOL, f"layer output error {err:.3e} (against the oracle for the GPU's h codes)"
    stats["y_err"] = err
    # against the oracle's own output: asserted for every position whose h
    # codes all equal the oracle's.  Where the GPU's fp32 h fell on the other
    # side of a Q8_0 rounding boundary (both codes are quantisations of h
    # within its fp32 error; checked above to be exactly such steps), one
    # code step can move y by more than 1e-3 of max|y| on narrow layers; those
    # positions are held to the adjusted bound and the elementwise bound.
    stats["y_err_unadjusted"] = normwise_err(y_g, ref["y"])
    stats["positions_with_h_step"] = int(stepped.sum())
    clean = ~stepped
    stats["y_err_unadjusted_no_step"] = normwise_err(y_g[clean], ref["y"][clean])
    assert stats["y_err_unadjusted_no_step"] <= Y_TOL, \
        f"layer output error {stats['y_err_unadjusted_no_step']:.3e} against the oracle's own output"
    stats["y_err_elementwise_rms_floor"] = elementwise_err(y_g, ref["y"])
    dy = np.abs(y_g.astype(np.float64) - ref["y"])
    assert np.all(dy <= bound + 1e-30), f"elementwise output bound exceeded by {(dy - bound).max():.3e}"
    return stats
