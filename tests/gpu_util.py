"""Helpers for the GPU parity tests: build caches on the device through the C ABI
and on the host through the oracle from the same seeded inputs, and compare.

No value computed by the CUDA path is ever fed to the oracle: device caches are
either built by the library from the synthetic tokens (and compared with the
oracle's own cache built from the same tokens), or filled with planes the
oracle quantised from synthetic rows.
"""
import multiprocessing as mp

import numpy as np
import torch

import oracle as O
from compressed_sparse_kv_05_b300 import dsv4, synth

DEV = "cuda"


def to_dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def to_host(t, dtype=None):
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


# ----------------------------------------------------------------------------- comparisons


def row_rel_err(got, ref):
    """max_d |g - o| / max_d |o| per row (last axis); 0 for an all-zero reference row equal to got."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.abs(got - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), num)


def _near_boundary(q, encode, delta):
    """True where an encoder's decision flips between q - delta and q + delta
    (delta: absolute, broadcastable to q)."""
    q = np.asarray(q, np.float64)
    d = np.abs(np.asarray(delta, np.float64)) + np.abs(q) * 2.0 ** -22
    return encode((q - d).astype(np.float32)) != encode((q + d).astype(np.float32))


def pooling_error_bound(oc, name):
    """Absolute bound [n_blocks][C] on the difference between a pooled value the
    kernels compute in fp32 and the oracle's float64 value rounded to fp32, for
    stream `name` ("k", "v" or "u") of an oracle cache from oracle_stream_cache.

    Per block and channel, with weights w_i = softmax_i(l_i), l_i = z_i + b_i:
    the fp32 side rounds l_i (2^-24 |l_i|), subtracts the block's max logit
    (2^-24 |l_i - max|) and takes exp (2 ulp = 2^-22): a relative error e_i on
    each weight; it then sums m weights and m products (2^-24 of the running
    sum each time) and divides once (2^-24). The oracle rounds once (2^-24).
    So |y_gpu - y_oracle| <= ((2m + 2) 2^-24 + 2 max_i e_i) A + 2^-23 |y| with
    A = sum_i w_i |x_i|, computed here in float64 from the same inputs."""
    ratio = oc["ratio"]
    x = np.abs(O.bf16_decode(oc["tokens"][name]))
    z = O.bf16_decode(oc["tokens"]["zu" if name == "u" else "z"])
    bias = np.asarray(oc["bias_u" if name == "u" else "bias"], np.float32).astype(np.float64)
    nb = x.shape[0] // ratio
    C = x.shape[1]
    x = x[: nb * ratio].reshape(nb, ratio, C)
    l = z[: nb * ratio].reshape(nb, ratio, C) + bias[None]
    mx = l.max(axis=1, keepdims=True)
    w = np.exp(l - mx)
    w /= w.sum(axis=1, keepdims=True)
    A = (w * x).sum(axis=1)
    e = (2.0 ** -22 + (np.abs(l) + np.abs(l - mx)) * 2.0 ** -24).max(axis=1)
    y = np.abs(oc["pooled_" + name]).astype(np.float64)
    return ((2 * ratio + 2) * 2.0 ** -24 + 2 * e) * A + 2.0 ** -23 * y


def compare_fp8_entries(g_codes, g_scale, o_codes, o_scale, o_pooled, d_nope, delta, max_frac=1e-3):
    """Comparison of FP8 entries built by two sides that pool in different
    precision: a pooled value may differ by up to `delta` (absolute, per
    element, from pooling_error_bound), so the row's amax, and with it the
    scale amax/448, may differ in its last bits (in most rows at ratio 128).
      * every row's scale must lie within the pooling bound of the oracle's;
      * every code must be the oracle's encoding of its own pooled value divided
        by the row's stored scale, except where that quotient lies within
        delta/scale of a rounding boundary; there it must be the code of one of
        the two sides of the boundary. Such codes are at most max_frac of all.
    Returns (codes at a rounding boundary, rows whose scale differs in its last bits)."""
    g_codes = np.asarray(g_codes).reshape(-1, d_nope)
    g_scale = np.asarray(g_scale, np.float32).reshape(-1)
    o_scale = np.asarray(o_scale, np.float32).reshape(-1)
    y = np.asarray(o_pooled, np.float32).reshape(-1, o_pooled.shape[-1])[:, :d_nope].astype(np.float64)
    dl = np.asarray(delta, np.float64).reshape(y.shape[0], -1)[:, :d_nope]
    amax_idx = np.abs(y).argmax(axis=1)
    d_amax = dl[np.arange(y.shape[0]), amax_idx]
    diff_s = np.abs(g_scale.astype(np.float64) - o_scale.astype(np.float64))
    assert (diff_s <= d_amax / 448 + 2.0 ** -20 * o_scale).all(), "scale differs beyond the pooling bound"
    zero = g_scale == 0
    assert not g_codes[zero].any(), "a zero scale with non-zero codes"
    s = np.where(zero, 1.0, g_scale.astype(np.float64))[:, None]
    q = y / s
    dq = dl / s
    want = O.e4m3_encode(q.astype(np.float32))
    want[zero] = 0
    rows, cols = np.nonzero(g_codes != want)
    if rows.size:
        qq, dd = q[rows, cols], dq[rows, cols]
        assert _near_boundary(qq, O.e4m3_encode, dd).all(), "FP8 code differs away from a rounding boundary"
        # the stored code must lie between the codes of the band's two ends
        lo = O.e4m3_decode(O.e4m3_encode((qq - dd - np.abs(qq) * 2.0 ** -22).astype(np.float32)))
        hi = O.e4m3_decode(O.e4m3_encode((qq + dd + np.abs(qq) * 2.0 ** -22).astype(np.float32)))
        gv = O.e4m3_decode(g_codes[rows, cols])
        assert ((gv >= lo) & (gv <= hi)).all(), "FP8 code outside the pooling band"
    assert rows.size <= max(8, max_frac * g_codes.size), rows.size
    n_scale = int((g_scale != o_scale).sum())
    same = g_scale == o_scale
    assert np.array_equal(g_codes[same & ~np.isin(np.arange(y.shape[0]), rows)],
                          np.asarray(o_codes).reshape(-1, d_nope)[same & ~np.isin(np.arange(y.shape[0]), rows)])
    print(f"fp8 entries: {g_codes.shape[0]} rows, {n_scale} whose scale differs in its last bits "
          f"(max relative {(diff_s / np.maximum(o_scale, 1e-38)).max():.2e}), {rows.size} codes at a rounding boundary")
    return rows.size, n_scale


def compare_fp4_rows(g_codes, g_scales, o_codes, o_scales, o_pooled, delta, max_frac=1e-3):
    """As compare_fp8_entries for FP4 rows (per-16 e4m3 scales)."""
    R = o_pooled.shape[0]
    C = o_pooled.shape[1]
    g_codes = np.asarray(g_codes).reshape(R, C // 2)
    o_codes = np.asarray(o_codes).reshape(R, C // 2)
    g_scales = np.asarray(g_scales).reshape(R, C // 16)
    o_scales = np.asarray(o_scales).reshape(R, C // 16)
    y = np.asarray(o_pooled, np.float32).reshape(R, C // 16, 16).astype(np.float64)
    dl = np.asarray(delta, np.float64).reshape(R, C // 16, 16)
    amax6 = np.abs(y).max(axis=2) / 6.0
    sdiff = g_scales != o_scales
    if sdiff.any():
        assert _near_boundary(amax6[sdiff], O.e4m3_encode, dl.max(axis=2)[sdiff] / 6.0).all(), \
            "FP4 scale differs away from a boundary"
    gn = np.stack([g_codes & 0xF, g_codes >> 4], axis=-1).reshape(R, C // 16, 16)
    on = np.stack([o_codes & 0xF, o_codes >> 4], axis=-1).reshape(R, C // 16, 16)
    diff = (gn != on) & ~sdiff[:, :, None]
    r, b, i = np.nonzero(diff)
    if r.size:
        s = O.e4m3_decode(o_scales[r, b]).astype(np.float64)
        assert _near_boundary(y[r, b, i] / s, O.e2m1_encode, dl[r, b, i] / s).all(), \
            "FP4 code differs away from a rounding boundary"
    assert r.size + int(sdiff.sum()) * 16 <= max(8, max_frac * gn.size), (r.size, int(sdiff.sum()))
    print(f"fp4 rows: {R} rows, {int(sdiff.sum())} block scales and {r.size} codes at a rounding boundary")
    return r.size, int(sdiff.sum())


def compare_bf16(g_bits, o_bits, o_pooled, delta, max_frac=1e-3):
    """bf16 bytes identical except where the oracle's pooled value lies within
    the pooling bound `delta` of a bf16 rounding boundary."""
    g = np.asarray(g_bits).reshape(-1)
    o = np.asarray(o_bits).reshape(-1)
    y = np.asarray(o_pooled, np.float32).reshape(-1)
    dl = np.asarray(delta, np.float64).reshape(-1)
    diff = g != o
    if diff.any():
        assert _near_boundary(y[diff], O.bf16_encode, dl[diff]).all(), "bf16 differs away from a rounding boundary"
    assert diff.sum() <= max(8, max_frac * g.size)
    print(f"bf16: {g.size} values, {int(diff.sum())} at a rounding boundary")
    return int(diff.sum())


def check_topk(g_topk, o_scores, o_topk, k, gap_rel=1e-6):
    """Top-k set parity: identical, except when the oracle's k-th score gap is
    below gap_rel relative; then every differing member must lie in the tied
    boundary band. Order must be ascending with -1 padding at the end."""
    g = np.asarray(g_topk)
    valid = g[g >= 0]
    assert (np.diff(valid) > 0).all(), "top-k not strictly ascending"
    assert (g[len(valid):] == -1).all()
    if np.array_equal(g, o_topk):
        return 0
    gap = O.topk_boundary_gap(o_scores, k)
    assert gap < gap_rel, f"top-k differs with boundary gap {gap}"
    kth = np.sort(o_scores)[::-1][k - 1]
    band = np.abs(o_scores - kth) <= gap_rel * abs(kth) * 4
    sym = set(valid.tolist()) ^ set(o_topk[o_topk >= 0].tolist())
    assert all(band[i] for i in sym)
    return len(sym)


# ----------------------------------------------------------------------------- caches built by the library from tokens


def gpu_stream_cache(layer, tag, layer_id, n_tokens, chunks, capacity=None):
    """Append synthetic tokens [0, n_tokens) in the given chunk sizes (cycled)
    through dsv4_compress_append. Returns (desc, cache)."""
    cap = capacity if capacity is not None else max(1, n_tokens // layer.ratio + 1)
    desc = dsv4.layer_desc(layer, cap)
    cache = dsv4.Cache(desc)
    b = to_dev(synth.position_bias(tag, layer_id, layer, "b"))
    bu = to_dev(synth.position_bias(tag, layer_id, layer, "bu")) if desc.idx_dim else None
    t0, ci = 0, 0
    while t0 < n_tokens:
        t1 = min(n_tokens, t0 + chunks[ci % len(chunks)])
        ci += 1
        toks = {k: to_dev(v) for k, v in synth.token_stream(tag, layer_id, layer, layer.batch, t0, t1).items()}
        dsv4.dsv4_compress_append(desc, cache, t1 - t0, toks["k"], toks.get("v"), toks["z"], b,
                                  toks.get("u"), toks.get("zu"), bu)
        t0 = t1
    torch.cuda.synchronize()
    return desc, cache


def oracle_stream_cache(layer, tag, layer_id, n_tokens, seq):
    toks = synth.token_stream(tag, layer_id, layer, layer.batch, 0, n_tokens)
    b = synth.position_bias(tag, layer_id, layer, "b")
    bu = synth.position_bias(tag, layer_id, layer, "bu") if layer.idx_dim else None
    c = O.build_cache(toks["k"][seq], toks["z"][seq], b, layer.ratio, layer.d_nope, layer.window,
                      toks["v"][seq] if layer.separate_v else None,
                      toks["u"][seq] if layer.idx_dim else None, toks["zu"][seq] if layer.idx_dim else None, bu)
    D = layer.dim
    W = layer.window
    ring = np.zeros((max(W, 1), D), np.uint16)
    for s, tok in c["win_k"].items():
        ring[s] = tok
    c["ring_k"] = ring
    if layer.separate_v:
        ringv = np.zeros((max(W, 1), D), np.uint16)
        for s, tok in c["win_v"].items():
            ringv[s] = tok
        c["ring_v"] = ringv
    c["tokens"] = {k: v[seq] for k, v in toks.items()}
    c["ratio"], c["bias"], c["bias_u"] = layer.ratio, b, bu
    return c


# ----------------------------------------------------------------------------- caches drawn directly


def _oracle_direct_planes(args):
    tag, layer_id, layer, seq = args
    rows = synth.direct_rows(tag, layer_id, layer, seq)
    out = {}
    out["k_nope"], out["k_scale"], out["k_rope"] = O.quantize_kv_rows(rows["kv"], layer.d_nope)
    if layer.separate_v:
        out["v_nope"], out["v_scale"], out["v_rope"] = O.quantize_kv_rows(rows["v"], layer.d_nope)
    if layer.kind == "csa":
        out["idx_codes"], out["idx_scales"] = O.quantize_fp4_rows(rows["idx"])
        out["planted"] = rows["planted"]
    win = synth.window_tokens(tag, layer_id, layer, seq)
    W, n = layer.window, layer.n_tokens
    pos = np.arange(n - min(W, n), n)
    ring = np.zeros((max(W, 1), layer.dim), np.uint16)
    ring[pos % max(W, 1)] = win["k"]
    out["ring_k"] = ring
    if layer.separate_v:
        ringv = np.zeros((max(W, 1), layer.dim), np.uint16)
        ringv[pos % max(W, 1)] = win["v"]
        out["ring_v"] = ringv
    return out


def oracle_direct_planes(layer, tag, layer_id, seqs, processes=None):
    """Oracle-quantised planes of directly drawn caches for the given sequences
    (a spawn process pool when several are asked for)."""
    args = [(tag, layer_id, layer, s) for s in seqs]
    if processes is None or processes <= 1 or len(args) == 1:
        return [_oracle_direct_planes(a) for a in args]
    with mp.get_context("spawn").Pool(processes) as pool:
        return pool.map(_oracle_direct_planes, args)


def gpu_cache_from_planes(layer, planes, capacity=None, extra=0):
    """Device cache holding the given per-sequence oracle planes, n_tokens set."""
    cap = capacity if capacity is not None else layer.capacity(extra)
    desc = dsv4.layer_desc(layer, cap)
    cache = dsv4.Cache(desc)
    n_c = layer.n_comp
    for b, p in enumerate(planes):
        cache.k_nope[b, :n_c] = to_dev(p["k_nope"])
        cache.k_scale[b, :n_c] = to_dev(p["k_scale"])
        cache.k_rope[b, :n_c] = to_dev(p["k_rope"])
        cache.win_k[b] = to_dev(p["ring_k"])
        if layer.separate_v:
            cache.v_nope[b, :n_c] = to_dev(p["v_nope"])
            cache.v_scale[b, :n_c] = to_dev(p["v_scale"])
            cache.v_rope[b, :n_c] = to_dev(p["v_rope"])
            cache.win_v[b] = to_dev(p["ring_v"])
        if layer.kind == "csa" and "idx_codes" in p:
            cache.idx_codes[b, :n_c] = to_dev(p["idx_codes"])
            cache.idx_scales[b, :n_c] = to_dev(p["idx_scales"])
    cache.n_tokens.fill_(layer.n_tokens)
    torch.cuda.synchronize()
    return desc, cache


def planes_from_rows(layer, kv, win, idx=None, v=None, win_v=None):
    """Oracle-quantised planes of one sequence from given pooled rows: kv (and v)
    float32 [n_c][D], window tokens win (and win_v) bf16 [min(W, n)][D] oldest
    first, indexer rows idx float32 [n_c][Di] for CSA."""
    out = {}
    out["k_nope"], out["k_scale"], out["k_rope"] = O.quantize_kv_rows(kv, layer.d_nope)
    if v is not None:
        out["v_nope"], out["v_scale"], out["v_rope"] = O.quantize_kv_rows(v, layer.d_nope)
    if idx is not None:
        out["idx_codes"], out["idx_scales"] = O.quantize_fp4_rows(idx)
    W, n = layer.window, layer.n_tokens
    pos = np.arange(n - min(W, n), n)
    for name, rows in (("ring_k", win), ("ring_v", win_v)):
        if rows is None:
            continue
        ring = np.zeros((max(W, 1), layer.dim), np.uint16)
        ring[pos % max(W, 1)] = rows
        out[name] = ring
    return out


def oracle_attend_planes(layer, p, q, sel):
    """Oracle attention of one sequence over planes (sel None: every entry, HCA)."""
    args = (layer.n_tokens, layer.ratio, layer.window, p["k_nope"], p["k_scale"], p["k_rope"], p["ring_k"])
    if layer.separate_v:
        args += (p["v_nope"], p["v_scale"], p["v_rope"], p["ring_v"])
    if sel is None:
        return O.hca_attend(q, np.float32(layer.sm_scale), *args)
    return O.csa_attend(q, np.float32(layer.sm_scale), sel, *args)


def check_pending(cache, oc, layer, b):
    """The open block's tokens (and gates) sit in the pending planes at slot t % ratio."""
    toks = oc["tokens"]
    names = [("pend_k", "k"), ("pend_z", "z")]
    if layer.separate_v:
        names.append(("pend_v", "v"))
    if layer.idx_dim:
        names += [("pend_u", "u"), ("pend_zu", "zu")]
    for plane, name in names:
        got = to_host(getattr(cache, plane), np.uint16)[b]
        for slot, t in oc["pending"].items():
            assert np.array_equal(got[slot, :toks[name].shape[1]], toks[name][t]), (plane, slot, t)
