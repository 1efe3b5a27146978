"""The parity harness's un-permutation of the library's activation layouts,
checked against the orders the C header states (no GPU needed)."""
import numpy as np

from helpers import unpermute_int2, unpermute_int4


def test_unpermute_int4_inverts_the_stated_order():
    # stored position s holds natural element order[s] within each group of 8
    order = [0, 2, 4, 6, 1, 3, 5, 7]
    nat = np.arange(64)
    stored = nat.reshape(-1, 8)[:, order].reshape(-1)
    assert np.array_equal(unpermute_int4(stored), nat)


def test_unpermute_int2_inverts_the_stated_order():
    # within each group of 16: 0,4,8,12, 1,5,9,13, 2,6,10,14, 3,7,11,15
    order = [0, 4, 8, 12, 1, 5, 9, 13, 2, 6, 10, 14, 3, 7, 11, 15]
    nat = np.arange(96).reshape(3, 32)
    stored = nat.reshape(3, -1, 16)[..., order].reshape(3, 32)
    assert np.array_equal(unpermute_int2(stored), nat)
    # the stored order pairs the m-th 2-bit field of packed bytes 0..3 with one
    # 4-byte activation word: word m holds elements m, 4+m, 8+m, 12+m
    assert stored[0, 4:8].tolist() == [1, 5, 9, 13]


def _oracle_observables(shape, x, wr, bias, get_record):
    """The observables the GPU parity check reads, filled from the oracle."""
    import oracle
    idx, w = oracle.route(oracle.router_logits(x, wr), bias, shape)
    ref = oracle.moe_forward(shape, get_record, x, idx, w, keep_pairs=True)
    tabs = ref["tables"]
    T, k = idx.shape
    P = T * k + shape.n_shared * T
    imax = max(shape.inter, shape.shared_inter)
    qh = np.zeros((P, imax), np.int8)
    dh = np.zeros((P, imax // 32), np.float32)
    acc_gu = np.zeros((P, 2, imax, shape.hidden // 32), np.int32)
    acc_d = np.zeros((P, shape.hidden, imax // 32), np.int32)
    where = {}
    for (kind, e), pr in ref["pairs"].items():
        for n, t in enumerate(pr["tokens"]):
            p = int(tabs["slot"][t, pr["js"][n]]) if kind == "routed" else \
                int(tabs["offsets"][tabs["uniq"].size + e] + t)
            qh[p] = pr["qh"][n]
            dh[p] = pr["dh"][n]
            acc_gu[p, 0], acc_gu[p, 1], acc_d[p] = pr["acc_g"][n], pr["acc_u"][n], pr["acc_d"][n]
            where[(kind, e, n)] = (p, int(t), float(w[t, pr["js"][n]]) if kind == "routed" else 1.0)
    n_ent = tabs["counts"].size
    g = dict(status=0, idx=idx, w=w.astype(np.float32), y=ref["y"].astype(np.float32), n_entries=n_ent,
             entry_expert=np.concatenate([tabs["uniq"], shape.n_experts + np.arange(shape.n_shared)]),
             entry_count=tabs["counts"], entry_offset=tabs["offsets"], pair_token=tabs["pair_token"],
             slot=tabs["slot"], qx=ref["qx"], dx=ref["dx"], qh=qh, dh=dh, acc_gu=acc_gu, acc_d=acc_d)
    return g, ref, where


def test_parity_check_accepts_only_admissible_h_code_steps():
    """The output tolerance is applied after accounting for a +-1 step of a
    requantised h code that sits on a rounding boundary (both codes are
    admissible); a step at a unique code, or an output error without a step,
    still fails."""
    import pytest
    from types import SimpleNamespace
    import oracle
    import synth
    from helpers import margin_batch
    try:
        from gpu_harness import check_parity
    except (ImportError, OSError) as exc:  # the harness loads the library (built by build())
        pytest.skip(f"library not built: {exc}")
    shape, seed = synth.TINY_INT2, 10
    routed = [synth.expert_record(shape, seed, 0, "routed", e) for e in range(shape.n_experts)]
    shared = [synth.expert_record(shape, seed, 0, "shared", 0)]
    get = lambda kind, e: routed[e] if kind == "routed" else shared[e]
    wr, bias = synth.router_weight(shape, seed), synth.router_bias(shape, seed)
    x, _, _ = margin_batch(shape, seed, ("int2", 33), 33, wr, bias)
    layer = SimpleNamespace(shape=shape, router_w=wr, bias=bias, get_record=get)
    g, ref, where = _oracle_observables(shape, x, wr, bias, get)
    check_parity(layer, x, g)

    # the non-unique code whose one-step change moves y the most
    best = None
    for (kind, e), pr in ref["pairs"].items():
        rec, sc = get(kind, e)
        wd = oracle.unpack_weight_rows(rec[2 * shape.inter * shape.row_bytes(shape.hidden):],
                                       shape.hidden, shape.inter, 2).astype(np.float64)
        s_d = sc[2 * shape.inter:2 * shape.inter + shape.hidden].astype(np.float64)
        for n in range(len(pr["tokens"])):
            p, t, wt = where[(kind, e, n)]
            for i in np.flatnonzero(~pr["qh_stable"][n]):
                dy = wt * s_d * float(pr["dh"][n][i // 32]) * wd[:, i]
                r = np.abs(dy).max() / np.abs(ref["y"][t]).max()
                if best is None or r > best[0]:
                    best = (r, p, t, i, dy, pr["qh_stable"][n], wd[:, i])
    r, p, t, i, dy, stable, wcol = best
    assert r > 1e-3          # a step here alone exceeds the output tolerance
    step = 1 if g["qh"][p, i] < 127 else -1
    gf = dict(g, qh=g["qh"].copy(), y=g["y"].copy(), acc_d=g["acc_d"].copy())
    gf["qh"][p, i] += step
    gf["acc_d"][p, :, i // 32] += (step * wcol).astype(np.int32)   # the down dots of the stepped block
    gf["y"][t] = (ref["y"][t] + step * dy).astype(np.float32)
    check_parity(layer, x, gf)
    # a down block dot that differs where the codes agree is rejected
    gd = dict(g, acc_d=g["acc_d"].copy())
    gd["acc_d"][p, 3, (i // 32 + 1) % (shape.inter // 32)] += 1
    with pytest.raises(AssertionError, match="down block dots"):
        check_parity(layer, x, gd)

    # the same step at a unique code is rejected
    j = int(np.flatnonzero(stable)[0])
    gu = dict(g, qh=g["qh"].copy())
    gu["qh"][p, j] += 1 if gu["qh"][p, j] < 127 else -1
    with pytest.raises(AssertionError):
        check_parity(layer, x, gu)
    # an output error of the step's size without the step is rejected
    ge = dict(g, y=g["y"].copy())
    ge["y"][t] = (ref["y"][t] + step * dy).astype(np.float32)
    with pytest.raises(AssertionError):
        check_parity(layer, x, ge)
