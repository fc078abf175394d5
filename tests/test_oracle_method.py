"""Pins of the oracle's pooling, quantisation, indexer, top-k and attention
against closed forms, brute force, exact rational arithmetic, a library routine
(torch's scaled_dot_product_attention in float64) and the invariants the method
fixes. A plausible slip (dropped bias, transposed operand, wrong nibble order,
sign or tie rule) fails at least one of these."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from compressed_sparse_kv_05_b300 import accounting, synth
from compressed_sparse_kv_05_b300 import workloads as W


def bf16(a):
    return synth.bf16_bits(np.asarray(a, np.float32))


def rnd(seed, shape, std=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * std).astype(np.float32)


# ----------------------------------------------------------------------------- pooling

def test_pool_ratio1_is_identity():
    x = bf16(rnd(1, (7, 24)))
    y = O.pool_blocks(x, bf16(rnd(2, (7, 24))), rnd(3, (1, 24)), 1)
    assert np.array_equal(y, O.bf16_decode(x).astype(np.float32))


def test_pool_zero_gates_is_mean():
    x = bf16(rnd(4, (12, 16)))
    y = O.pool_blocks(x, bf16(np.zeros((12, 16))), np.zeros((4, 16), np.float32), 4)
    ref = O.bf16_decode(x).reshape(3, 4, 16).mean(axis=1)
    assert np.allclose(y, ref, rtol=1e-6, atol=1e-7)


def test_pool_ratio2_closed_form():
    x = bf16(rnd(5, (10, 8)))
    z = bf16(rnd(6, (10, 8)))
    b = rnd(7, (2, 8), 0.1)
    y = O.pool_blocks(x, z, b, 2)
    xd, zd = O.bf16_decode(x).reshape(5, 2, 8), O.bf16_decode(z).reshape(5, 2, 8)
    delta = (zd[:, 0] + b[0]) - (zd[:, 1] + b[1])
    sig = 1.0 / (1.0 + np.exp(-delta))
    ref = sig * xd[:, 0] + (1 - sig) * xd[:, 1]
    assert np.allclose(y, ref, rtol=1e-6, atol=1e-7)


def test_pool_identical_tokens_give_that_token():
    row = bf16(rnd(8, (1, 32)))
    x = np.repeat(row, 128, axis=0)
    y = O.pool_blocks(x, bf16(rnd(9, (128, 32))), rnd(10, (128, 32), 0.1), 128)
    assert np.array_equal(y[0], O.bf16_decode(row[0]).astype(np.float32))


def test_pool_bias_shift_invariance_and_bias_matters():
    x = bf16(rnd(11, (16, 8)))
    z = bf16(rnd(12, (16, 8)))
    b = rnd(13, (4, 8), 0.1)
    y0 = O.pool_blocks(x, z, b, 4)
    y1 = O.pool_blocks(x, z, b + rnd(14, (1, 8), 3.0), 4)   # same shift for every position of a channel
    # b + shift is rounded to fp32 (|error| <= 2**-21 in the logits), hence the tolerance
    assert np.allclose(y0, y1, rtol=2e-5, atol=2e-6)
    y2 = O.pool_blocks(x, z, b * 10, 4)                     # a different bias changes the weights
    assert not np.allclose(y0, y2, rtol=1e-3)


def test_pool_drops_incomplete_block():
    x = bf16(rnd(15, (11, 8)))
    y = O.pool_blocks(x, bf16(rnd(16, (11, 8))), rnd(17, (4, 8)), 4)
    assert y.shape == (2, 8)


# ----------------------------------------------------------------------------- quantisation

def test_kv_quant_exact_on_representable_rows():
    r = np.random.default_rng(18)
    R, dn, dr = 50, 64, 16
    codes = r.integers(0, 0x7F, size=(R, dn)).astype(np.uint8) | (r.integers(0, 2, (R, dn)).astype(np.uint8) << 7)
    codes[:, 5] = np.where(r.integers(0, 2, R) == 1, 0x7E, 0xFE)           # one +-448 per row
    s = np.exp2(r.integers(-20, 5, R)).astype(np.float32)                  # power-of-two scales
    y = np.concatenate([(O.e4m3_decode(codes) * s[:, None]).astype(np.float32),
                        O.bf16_decode(bf16(rnd(19, (R, dr)))).astype(np.float32)], axis=1)
    c2, s2, rope = O.quantize_kv_rows(y, dn)
    assert np.array_equal(s2, s)
    # -0 codes (0x80) legitimately re-encode as -0; compare decoded values and signs
    assert np.array_equal(O.e4m3_decode(c2), O.e4m3_decode(codes))
    assert np.array_equal(rope, bf16(y[:, dn:]))


def test_dequant_kv_rows_against_library_decode():
    """dequant_kv_rows against torch's own e4m3 and bf16 decodes, on entries
    whose row count, code dims and RoPE dims all differ and whose per-row scales
    all differ: each value is its code times its own row's scale, then the RoPE
    dims follow in order (a scale broadcast along the wrong axis, a row slip or
    a dropped RoPE block fails)."""
    r = np.random.default_rng(31)
    R, dn, dr = 37, 48, 16
    codes = r.integers(0, 256, size=(R, dn)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C                                   # no NaN codes
    s = (np.exp2(r.integers(-30, 10, R)) * r.choice([1.0, 1.25, 1.5, 1.75], R)).astype(np.float32)
    rope = bf16(rnd(32, (R, dr)))
    got = O.dequant_kv_rows(codes, s, rope)
    lib_codes = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    lib_rope = torch.from_numpy(rope.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    want = np.concatenate([lib_codes * s.astype(np.float64)[:, None], lib_rope], axis=1)
    assert got.shape == (R, dn + dr) and np.array_equal(got, want)
    # exactly representable rows come back unchanged through quantise -> dequantise
    codes2 = r.integers(0, 0x7F, size=(R, dn)).astype(np.uint8)
    codes2[:, 7] = 0x7E                                                    # each row reaches 448 * s
    s2 = np.exp2(r.integers(-24, 6, R)).astype(np.float32)
    y = np.concatenate([(torch.from_numpy(codes2).view(torch.float8_e4m3fn).to(torch.float64).numpy()
                         * s2.astype(np.float64)[:, None]).astype(np.float32),
                        O.bf16_decode(rope).astype(np.float32)], axis=1)
    assert np.array_equal(O.dequant_kv_rows(*O.quantize_kv_rows(y, dn)), y.astype(np.float64))


def test_kv_quant_zero_row_and_error_bound():
    y = rnd(20, (40, 80))
    y[3, :64] = 0.0
    c, s, _ = O.quantize_kv_rows(y, 64)
    assert s[3] == 0 and not c[3].any()
    deq = O.e4m3_decode(c) * s[:, None]
    amax = np.abs(y[:, :64]).max(axis=1)
    assert np.isclose(np.abs(deq).max(axis=1), amax, rtol=1e-6).all()
    big = np.abs(y[:, :64]) >= amax[:, None] * 2.0 ** -6 / 448 * 448   # normal range of the code grid
    err = np.abs(deq - y[:, :64])
    assert (err[big] <= np.abs(y[:, :64])[big] * 2.0 ** -4 * 1.0001).all()


def test_fp4_quant_exact_on_representable_rows_and_nibble_order():
    r = np.random.default_rng(21)
    R, C = 30, 64
    nib = r.integers(0, 16, size=(R, C)).astype(np.uint8)
    nib[:, ::16] = np.where(r.integers(0, 2, (R, C // 16)) == 1, 7, 15)     # one +-6 per block of 16
    sc = r.integers(0x20, 0x60, size=(R, C // 16)).astype(np.uint8)        # e4m3 scales, normal range
    y = (O.e2m1_decode(nib).reshape(R, C // 16, 16) * O.e4m3_decode(sc)[:, :, None]).reshape(R, C).astype(np.float32)
    codes, scales = O.quantize_fp4_rows(y)
    assert np.array_equal(scales, sc)
    assert np.array_equal(O.dequant_fp4_rows(codes, scales), y.astype(np.float64))
    assert np.array_equal(codes[:, 0] & 0xF, np.where(nib[:, 0] == 8, 0, nib[:, 0]) | (nib[:, 0] & 8))
    # element 1 sits in the high nibble of byte 0
    assert np.array_equal(O.e2m1_decode(codes[:, 0] >> 4), O.e2m1_decode(nib[:, 1]))


def test_fp4_quant_zero_block():
    y = rnd(22, (4, 32))
    y[1, 16:] = 0
    codes, scales = O.quantize_fp4_rows(y)
    assert scales[1, 1] == 0 and not codes[1, 8:].any()


# ----------------------------------------------------------------------------- indexer

def _fp4_rows(seed, R, C):
    return O.quantize_fp4_rows(rnd(seed, (R, C)))


def test_index_scores_exact_rational():
    Hi, Di, n = 3, 32, 9
    kc, ks = _fp4_rows(23, n, Di)
    q = bf16(rnd(24, (Hi, Di)))
    w = np.random.default_rng(25).uniform(0, 1, Hi).astype(np.float32)
    got = O.index_scores(kc, ks, q, w)
    qc, qs = O.quantize_fp4_rows(O.bf16_decode(q).astype(np.float32))

    def frac_rows(codes, scales):
        out = []
        for i in range(codes.shape[0]):
            row = []
            for j in range(codes.shape[1] * 2):
                byte = int(codes[i, j // 2])
                nibble = byte & 0xF if j % 2 == 0 else byte >> 4
                row.append(Fraction(float(O.e2m1_decode(np.array([nibble]))[0])) *
                           Fraction(float(O.e4m3_decode(np.array([scales[i, j // 16]], np.uint8))[0])))
            out.append(row)
        return out
    K, Q = frac_rows(kc, ks), frac_rows(qc, qs)
    for s in range(n):
        exact = sum(Fraction(float(w[h])) * max(Fraction(0), sum(a * b for a, b in zip(Q[h], K[s])))
                    for h in range(Hi))
        assert abs(Fraction(got[s]) - exact) <= abs(exact) * Fraction(1, 10 ** 14)


def test_index_scores_single_head_is_relu_dot():
    kc, ks = _fp4_rows(26, 20, 64)
    q = bf16(rnd(27, (1, 64)))
    got = O.index_scores(kc, ks, q, np.ones(1, np.float32))
    qd = O.dequant_fp4_rows(*O.quantize_fp4_rows(O.bf16_decode(q).astype(np.float32)))[0]
    ref = np.maximum(O.dequant_fp4_rows(kc, ks) @ qd, 0)
    assert np.array_equal(got, ref)
    assert (got == 0).any() and (got > 0).any()


# ----------------------------------------------------------------------------- top-k

@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force_with_ties(seed):
    r = np.random.default_rng(seed)
    n = int(r.integers(1, 40))
    k = int(r.integers(1, 12))
    scores = r.integers(0, 5, n).astype(np.float64)       # many exact ties
    got = O.topk_blocks(scores, k)
    brute = sorted(range(n), key=lambda i: (-scores[i], i))[:k]
    ref = sorted(brute) + [-1] * (k - len(brute))
    assert got.tolist() == ref


def test_topk_gap():
    assert O.topk_boundary_gap([5.0, 4.0, 4.0], 2) == 0.0
    assert O.topk_boundary_gap([5.0, 4.0, 2.0], 2) == 0.5
    assert O.topk_boundary_gap([5.0], 2) == np.inf


# ----------------------------------------------------------------------------- attention

def test_attend_matches_sdpa_fp64():
    H, N, D, Dv = 5, 37, 24, 16
    q = bf16(rnd(30, (H, D)))
    K = rnd(31, (N, D)).astype(np.float64)
    V = rnd(32, (N, Dv)).astype(np.float64)
    sc = np.float32(1 / math.sqrt(D))
    out, lse = O.attend(q, K, V, sc)
    qt = torch.from_numpy(O.bf16_decode(q))[None, :, None, :]          # [1][H][1][D]
    kt = torch.from_numpy(K)[None, None].expand(1, H, N, D)
    vt = torch.from_numpy(V)[None, None].expand(1, H, N, Dv)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=float(sc))[0, :, 0].numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-13)
    s = float(sc) * O.bf16_decode(q) @ K.T
    assert np.allclose(lse, np.log(np.exp(s).sum(axis=1)), rtol=1e-13)


def test_attend_single_key_and_equal_scores():
    q = bf16(rnd(33, (3, 8)))
    v = rnd(34, (1, 6)).astype(np.float64)
    out, _ = O.attend(q, rnd(35, (1, 8)).astype(np.float64), v, 0.3)
    assert np.allclose(out, np.repeat(v, 3, axis=0), rtol=1e-15)
    K = np.repeat(rnd(36, (1, 8)).astype(np.float64), 10, axis=0)
    V = rnd(37, (10, 6)).astype(np.float64)
    out, lse = O.attend(q, K, V, 0.3)
    assert np.allclose(out, np.repeat(V.mean(axis=0, keepdims=True), 3, axis=0), rtol=1e-13)


def test_attend_empty_set():
    out, lse = O.attend(bf16(rnd(38, (2, 4))), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert not out.any() and np.all(np.isneginf(lse))


def test_union_softmax_equals_lse_merge():
    q = bf16(rnd(39, (4, 16)))
    Ka, Kb = rnd(40, (20, 16)).astype(np.float64), rnd(41, (7, 16)).astype(np.float64)
    Va, Vb = rnd(42, (20, 16)).astype(np.float64), rnd(43, (7, 16)).astype(np.float64)
    oa, la = O.attend(q, Ka, Va, 0.25)
    ob, lb = O.attend(q, Kb, Vb, 0.25)
    om, lm = O.lse_merge([oa, ob], [la, lb])
    ou, lu = O.attend(q, np.concatenate([Ka, Kb]), np.concatenate([Va, Vb]), 0.25)
    assert np.allclose(om, ou, rtol=1e-12, atol=1e-14) and np.allclose(lm, lu, rtol=1e-13)
    oe, le = O.lse_merge([oa, np.zeros_like(oa)], [la, np.full(4, -np.inf)])   # an empty partial
    assert np.allclose(oe, oa) and np.allclose(le, la)


def _small_cache(seed, n, ratio, d_nope, d_rope, window, separate_v, idx_dim=0):
    D = d_nope + d_rope
    k = bf16(rnd(seed, (n, D)))
    z = bf16(rnd(seed + 1, (n, D)))
    b = rnd(seed + 2, (ratio, D), 0.1)
    v = bf16(rnd(seed + 3, (n, D))) if separate_v else None
    u = zu = bu = None
    if idx_dim:
        u, zu, bu = bf16(rnd(seed + 4, (n, idx_dim))), bf16(rnd(seed + 5, (n, idx_dim))), rnd(seed + 6, (ratio, idx_dim), 0.1)
    c = O.build_cache(k, z, b, ratio, d_nope, window, v, u, zu, bu)
    ring = np.zeros((window, D), np.uint16)
    for s_, tok in c["win_k"].items():
        ring[s_] = tok
    c["ring_k"] = ring
    if separate_v:
        ringv = np.zeros((window, D), np.uint16)
        for s_, tok in c["win_v"].items():
            ringv[s_] = tok
        c["ring_v"] = ringv
    return c, k, v


def test_csa_ratio1_all_selected_no_window_is_full_attention():
    n, dn, dr = 48, 32, 16
    c, k, _ = _small_cache(50, n, 1, dn, dr, 0, False)
    q = bf16(rnd(51, (6, dn + dr)))
    out, lse = O.csa_attend(q, 0.2, np.arange(n), n, 1, 0, c["k_nope"], c["k_scale"], c["k_rope"], None)
    codes, scale, rope = O.quantize_kv_rows(O.bf16_decode(k).astype(np.float32), dn)
    Kfull = np.concatenate([O.e4m3_decode(codes) * scale.astype(np.float64)[:, None], O.bf16_decode(rope)], axis=1)
    qt = torch.from_numpy(O.bf16_decode(q))[None, :, None, :]
    kt = torch.from_numpy(Kfull)[None, None].expand(1, 6, n, dn + dr)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, kt, scale=float(np.float32(0.2)))[0, :, 0].numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_csa_permutation_invariance_and_padding():
    n = 64 * 4 + 3
    c, _, _ = _small_cache(60, n, 4, 32, 16, 8, True)
    q = bf16(rnd(61, (3, 48)))
    sel = np.array([5, 9, 0, 63, 17], np.int32)
    args = (n, 4, 8, c["k_nope"], c["k_scale"], c["k_rope"], c["ring_k"], c["v_nope"], c["v_scale"], c["v_rope"], c["ring_v"])
    o1, l1 = O.csa_attend(q, 0.1, sel, *args)
    o2, l2 = O.csa_attend(q, 0.1, np.concatenate([sel[::-1], [-1, -1]]), *args)
    assert np.allclose(o1, o2, rtol=1e-13) and np.allclose(l1, l2, rtol=1e-14)
    with pytest.raises(ValueError):
        O.csa_attend(q, 0.1, np.array([n // 4]), *args)


def test_csa_is_merge_of_window_and_selected_partials():
    n = 200
    c, k, v = _small_cache(70, n, 4, 32, 16, 16, True)
    q = bf16(rnd(71, (2, 48)))
    sel = np.array([1, 7, 30, 49], np.int32)
    o, l = O.csa_attend(q, 0.15, sel, n, 4, 16, c["k_nope"], c["k_scale"], c["k_rope"], c["ring_k"],
                        c["v_nope"], c["v_scale"], c["v_rope"], c["ring_v"])
    Ks = O.dequant_kv_rows(c["k_nope"][sel], c["k_scale"][sel], c["k_rope"][sel])
    Vs = O.dequant_kv_rows(c["v_nope"][sel], c["v_scale"][sel], c["v_rope"][sel])
    oa, la = O.attend(q, Ks, Vs, 0.15)
    ob, lb = O.attend(q, O.bf16_decode(k[n - 16:]), O.bf16_decode(v[n - 16:]), 0.15)   # window = last 16 raw tokens
    om, lm = O.lse_merge([oa, ob], [la, lb])
    assert np.allclose(o, om, rtol=1e-12, atol=1e-14) and np.allclose(l, lm, rtol=1e-13)


def test_hca_equals_csa_with_every_entry_selected():
    n = 128 * 5 + 17
    c, _, _ = _small_cache(80, n, 128, 32, 16, 32, False)
    q = bf16(rnd(81, (4, 48)))
    a = O.hca_attend(q, 0.1, n, 128, 32, c["k_nope"], c["k_scale"], c["k_rope"], c["ring_k"])
    b = O.csa_attend(q, 0.1, np.arange(5)[::-1], n, 128, 32, c["k_nope"], c["k_scale"], c["k_rope"], c["ring_k"])
    assert np.allclose(a[0], b[0], rtol=1e-13)


def test_window_ring_holds_last_tokens():
    n, W = 23, 8
    k = np.arange(n, dtype=np.uint16)[:, None].repeat(4, axis=1)
    c = O.build_cache(k, k, np.zeros((4, 4), np.float32), 4, 2, W)
    assert sorted(c["ring_slots"].values()) == list(range(n - W, n))
    for slot, tok in c["ring_slots"].items():
        assert slot == tok % W and c["win_k"][slot][0] == tok
    assert c["pending"] == {0: 20, 1: 21, 2: 22}


# ----------------------------------------------------------------------------- accounting

def test_kv_bytes_per_token_is_about_two_percent_of_gqa():
    gold = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "page_kv_ratio.txt")):
        if line.strip() and not line.startswith("#"):
            name, val = line.split()
            gold[name] = float(val)
    per_tok = np.mean([accounting.kv_bytes_per_token(l) for l in W.STACK_1M])
    ratio = per_tok / accounting.gqa_bf16_bytes_per_token()
    assert accounting.entry_bytes(W.STACK_CSA) == 580 and accounting.idx_key_bytes(W.STACK_CSA) == 72
    assert abs(per_tok - 83.8) < 0.1
    assert abs(ratio - gold["kv_ratio_vs_gqa8_bf16"]) < 0.005        # 2.05% against "about 2%"


def test_decode_step_bytes():
    assert accounting.decode_step_bytes(W.STACK_CSA) == 4 * (262144 * 72 + 64 * 128 * 2 + 64 * 4 + 512 * 580
                                                              + 128 * 512 * 2 + 64 * 512 * 2 + 64 * 512 * 4)
    assert accounting.decode_step_bytes(W.STACK_HCA) == 4 * (8192 * 580 + 128 * 512 * 2 + 64 * 512 * 6)


# ----------------------------------------------------------------------------- several queries per step

def _span(rows_bits, n, T, W):
    """Raw rows of the positions n - T - W + 1 .. n - 1 (zeros for negative positions)."""
    first = n - T - W + 1
    out = np.zeros((T + W - 1, rows_bits.shape[1]), np.uint16)
    for r in range(T + W - 1):
        if first + r >= 0:
            out[r] = rows_bits[first + r]
    return out


def _ring(cache, key, W, D):
    ring = np.zeros((W, D), np.uint16)
    for slot, tok in cache[key].items():
        ring[slot] = tok
    return ring


@pytest.mark.parametrize("n,T", [(90, 7), (9, 9), (41, 1), (130, 33)])
def test_multi_token_step_equals_single_token_decode_on_each_prefix(n, T):
    """Query t of a T-query step (position p = n - T + t) equals a single-token
    decode on the cache of its own prefix of p + 1 tokens, built and attended
    by the single-token functions: the same indexer scores, the same selection
    and the same attention (CSA and HCA); some queries see fewer blocks than
    the top-k, the first ones fewer tokens than the window."""
    W, ratio, dn, dr, Di, H, Hi, kk = 8, 4, 32, 16, 32, 3, 2, 5
    D = dn + dr
    k, z, v = bf16(rnd(90, (n, D))), bf16(rnd(91, (n, D))), bf16(rnd(92, (n, D)))
    u, zu = bf16(rnd(93, (n, Di))), bf16(rnd(94, (n, Di)))
    b, bu = rnd(95, (ratio, D), 0.1), rnd(96, (ratio, Di), 0.1)
    full = O.build_cache(k, z, b, ratio, dn, W, v, u, zu, bu)
    q, qi = bf16(rnd(97, (T, H, D))), bf16(rnd(98, (T, Hi, Di)))
    w = np.random.default_rng(99).uniform(0, 1, (T, Hi)).astype(np.float32)
    sm = np.float32(1 / np.sqrt(D))
    scores = O.index_scores_causal(full["idx_codes"], full["idx_scales"], qi, w, n, ratio)
    sel = np.stack([O.topk_blocks(sc, kk) for sc in scores])
    planes = (full["k_nope"], full["k_scale"], full["k_rope"], _span(k, n, T, W),
              full["v_nope"], full["v_scale"], full["v_rope"], _span(v, n, T, W))
    out, lse = O.multi_attend(q, sm, sel, n, ratio, W, *planes)
    outh, lseh = O.multi_attend(q, sm, None, n, ratio, W, *planes)
    assert out.shape == (T, H, D) and lse.shape == (T, H)
    for t, p in enumerate(O.query_positions(n, T)):
        pre = O.build_cache(k[:p + 1], z[:p + 1], b, ratio, dn, W, v[:p + 1], u[:p + 1], zu[:p + 1], bu)
        args = (p + 1, ratio, W, pre["k_nope"], pre["k_scale"], pre["k_rope"], _ring(pre, "win_k", W, D),
                pre["v_nope"], pre["v_scale"], pre["v_rope"], _ring(pre, "win_v", W, D))
        sc1 = O.index_scores(pre["idx_codes"], pre["idx_scales"], qi[t], w[t])
        assert np.array_equal(sc1, scores[t])
        assert np.array_equal(O.topk_blocks(sc1, kk), sel[t])
        o1, l1 = O.csa_attend(q[t], sm, sel[t], *args)
        assert np.allclose(o1, out[t], rtol=1e-12, atol=1e-14) and np.allclose(l1, lse[t], rtol=1e-13, atol=1e-13)
        oh, lh = O.hca_attend(q[t], sm, *args)
        assert np.allclose(oh, outh[t], rtol=1e-12, atol=1e-14) and np.allclose(lh, lseh[t], rtol=1e-13, atol=1e-13)


def test_multi_token_step_is_causal():
    """A query does not see the tokens after its own position: changing them
    (their raw rows and the blocks they complete) leaves its output unchanged,
    while changing a token inside its window changes it."""
    n, T, W, ratio, dn, dr = 64, 12, 6, 4, 32, 16
    D = dn + dr
    k, z = bf16(rnd(110, (n, D))), bf16(rnd(111, (n, D)))
    b = rnd(112, (ratio, D), 0.1)
    q = bf16(rnd(113, (T, 4, D)))
    t = 5
    p = n - T + t

    def run(kk):
        c = O.build_cache(kk, z, b, ratio, dn, W)
        return O.multi_attend(q, 0.2, None, n, ratio, W, c["k_nope"], c["k_scale"], c["k_rope"], _span(kk, n, T, W))

    base, _ = run(k)
    later = k.copy()
    later[p + 1:] = bf16(rnd(114, (n - p - 1, D)))
    after, _ = run(later)
    assert np.array_equal(after[:t + 1], base[:t + 1]) and not np.allclose(after[t + 1:], base[t + 1:])
    inside = k.copy()
    inside[p - 1] = bf16(rnd(115, (1, D)))
    changed, _ = run(inside)
    assert not np.allclose(changed[t], base[t]) and np.array_equal(changed[:t - 1], base[:t - 1])


# ----------------------------------------------------------------------------- projections and RoPE


def test_rope_position_zero_is_identity():
    x = rnd(120, (5, 64))
    assert np.array_equal(O.rope_rotate(x, np.zeros(5), 10000.0), x)


def test_rope_keeps_every_pair_norm():
    x = rnd(121, (7, 32)).astype(np.float64)
    y = O.rope_rotate(x, np.arange(7) * 977 + 3, 10000.0)
    nx = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
    ny = y[:, 0::2] ** 2 + y[:, 1::2] ** 2
    assert np.allclose(nx, ny, rtol=1e-12, atol=0)


def test_rope_scores_depend_on_relative_position_only():
    """<rope(q, m), rope(k, n)> = <rope(q, m - n), k>: the rotation composes by
    angle, so a score sees only the distance (and pins the sign convention: a
    rotation by -angle for one operand would break it)."""
    q, k = rnd(122, (1, 64)).astype(np.float64), rnd(123, (1, 64)).astype(np.float64)
    for m, n in [(5, 2), (1000, 37), (1 << 20, (1 << 20) - 129)]:
        lhs = (O.rope_rotate(q, [m], 500.0) * O.rope_rotate(k, [n], 500.0)).sum()
        rhs = (O.rope_rotate(q, [m - n], 500.0) * k).sum()
        assert abs(lhs - rhs) <= 1e-9 * (np.abs(q).sum() * np.abs(k).max())


def test_rope_pairs_are_adjacent_dims_with_geometric_frequencies():
    """A one-hot at dim 2i stays in dims (2i, 2i + 1) and turns by pos * base^(-2i/d):
    the first pair by pos radians, the middle pair (i = d/4) by pos / sqrt(base)."""
    d, base = 64, 10000.0
    for i, pos, ang in [(0, 1, 1.0), (0, 3, 3.0), (d // 4, 200, 200 / math.sqrt(base))]:
        e = np.zeros((1, d))
        e[0, 2 * i] = 1.0
        y = O.rope_rotate(e, [pos], base)[0]
        others = np.delete(y, [2 * i, 2 * i + 1])
        assert np.all(others == 0)
        assert abs(y[2 * i] - math.cos(ang)) < 1e-12 and abs(y[2 * i + 1] - math.sin(ang)) < 1e-12


def test_project_streams_one_hot_hidden_rows_pick_weight_columns():
    """Hidden rows with a single 1.0 select one weight column: the unrotated
    dims of x, all of z and zu, and the unrotated dims of u are that column's
    bf16 weights exactly; the rotated dims are its rotation at the token's position."""
    dn, dr, di, hdim = 8, 8, 16, 24
    D = dn + dr
    w = bf16(rnd(124, (2 * D + 2 * di, hdim)))
    cols = [0, 5, 23]
    h = np.zeros((3, hdim))
    for r, c in enumerate(cols):
        h[r, c] = 1.0
    pos = np.array([0, 7, 1 << 19])
    x, z, u, zu = O.project_streams(bf16(h), w, dn, dr, di, pos, 10000.0)
    wf = O.bf16_decode(w)
    for r, c in enumerate(cols):
        col = wf[:, c]
        assert np.array_equal(O.bf16_decode(x[r, :dn]), col[:dn])
        assert np.array_equal(O.bf16_decode(z[r]), col[D:2 * D])
        assert np.array_equal(O.bf16_decode(u[r, :di - dr]), col[2 * D:2 * D + di - dr])
        assert np.array_equal(O.bf16_decode(zu[r]), col[2 * D + di:])
        rx = O.rope_rotate(col[None, dn:D], [pos[r]], 10000.0)[0]
        ru = O.rope_rotate(col[None, 2 * D + di - dr:2 * D + di], [pos[r]], 10000.0)[0]
        assert np.array_equal(x[r, dn:], O.bf16_encode(rx))
        assert np.array_equal(u[r, di - dr:], O.bf16_encode(ru))


def test_project_streams_small_integers_are_exact_dot_products():
    """Integer hidden states and weights small enough that every dot product is
    an integer of magnitude < 256 (exact in bf16): the unrotated streams equal
    the dot products summed in Python integers."""
    dn, dr, di, hdim = 4, 4, 8, 6
    D = dn + dr
    rng = np.random.default_rng(125)
    h = rng.integers(-3, 4, (5, hdim))
    w = rng.integers(-3, 4, (2 * D + 2 * di, hdim))
    x, z, u, zu = O.project_streams(bf16(h.astype(np.float64)), bf16(w.astype(np.float64)), dn, dr, di,
                                    np.arange(5), 10000.0)
    for t in range(5):
        exact = [sum(int(h[t, c]) * int(w[n, c]) for c in range(hdim)) for n in range(w.shape[0])]
        assert O.bf16_decode(z[t]).tolist() == exact[D:2 * D]
        assert O.bf16_decode(x[t, :dn]).tolist() == exact[:dn]
        assert O.bf16_decode(zu[t]).tolist() == exact[2 * D + di:]
        assert O.bf16_decode(u[t, :di - dr]).tolist() == exact[2 * D:2 * D + di - dr]
