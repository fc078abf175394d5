"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
identical seeded inputs.

Bars: quantised bytes and top-k indices bit-exact except at the stated
rounding/tie exceptions; attention outputs and pooled fp32 values within 2e-3
max relative error per row (max_d |g - o| / max_d |o|)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from compressed_sparse_kv_05_b300 import dsv4, synth
from compressed_sparse_kv_05_b300 import workloads as W

from .gpu_util import (check_topk, compare_bf16, compare_fp4_rows, compare_fp8_entries, gpu_cache_from_planes,
                       gpu_stream_cache, oracle_direct_planes, oracle_stream_cache, pooling_error_bound, row_rel_err,
                       to_dev, to_host)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

TOL = 2e-3


# ----------------------------------------------------------------------------- formats and quantisers


def _wide_rows(seed, R, C):
    r = np.random.default_rng(seed)
    y = (r.standard_normal((R, C)) * np.exp2(r.uniform(-30, 30, (R, 1)))).astype(np.float32)
    y[0] = 0.0
    y[1, ::3] = -0.0
    y[2] = np.float32(1e-41)            # subnormal row
    return y


def test_quantize_kv_rows_bit_exact():
    for d_nope, d_rope in ((64, 64), (448, 64), (16, 0)):
        y = _wide_rows(d_nope, 3000, d_nope + d_rope)
        nope = torch.zeros((3000, d_nope), dtype=torch.uint8, device="cuda")
        scale = torch.zeros(3000, dtype=torch.float32, device="cuda")
        rope = torch.zeros((3000, max(d_rope, 8)), dtype=torch.int16, device="cuda")
        dsv4.dsv4_quantize_kv_rows(to_dev(y), 3000, d_nope, d_rope, nope, scale, rope)
        oc, os_, orope = O.quantize_kv_rows(y, d_nope)
        assert np.array_equal(to_host(nope), oc)
        assert np.array_equal(to_host(scale).view(np.uint32), os_.view(np.uint32))
        if d_rope:
            assert np.array_equal(to_host(rope, np.uint16)[:, :d_rope], orope)


def test_quantize_fp4_rows_bit_exact():
    for C in (64, 128, 256):
        y = _wide_rows(C + 1, 4000, C)
        codes = torch.zeros((4000, C // 2), dtype=torch.uint8, device="cuda")
        scales = torch.zeros((4000, C // 16), dtype=torch.uint8, device="cuda")
        dsv4.dsv4_quantize_fp4_rows(to_dev(y), 4000, C, codes, scales)
        oc, os_ = O.quantize_fp4_rows(y)
        assert np.array_equal(to_host(scales), os_)
        assert np.array_equal(to_host(codes), oc)


def test_hardware_conversions_match_oracle_encoders_sweep():
    """Rows whose amax is exactly 448 (resp. blocks whose amax is 6) have scale
    1, so the stored codes are the bare e4m3 (e2m1) conversions of the values:
    a sweep of ~4M values against the oracle's encoders, ties included."""
    r = np.random.default_rng(7)
    n_rows = 8192
    y = (r.standard_normal((n_rows, 512)) * np.exp2(r.uniform(-12, 8, (n_rows, 512)))).astype(np.float32)
    y = np.clip(y, -447.0, 447.0)
    grid = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((np.sort(grid)[1:] + np.sort(grid)[:-1]) / 2).astype(np.float32)
    y[:100, : mids.size] = mids[None]
    y[100:200, : mids.size] = -mids[None]
    y[:, 0] = 448.0
    nope = torch.zeros((n_rows, 512), dtype=torch.uint8, device="cuda")
    scale = torch.zeros(n_rows, dtype=torch.float32, device="cuda")
    dsv4.dsv4_quantize_kv_rows(to_dev(y), n_rows, 512, 0, nope, scale, None)
    assert (to_host(scale) == 1.0).all()
    assert np.array_equal(to_host(nope), O.e4m3_encode(y))
    # e2m1: blocks with one element equal to 6 -> scale e4m3(1) = 1
    f = (r.uniform(-6, 6, (n_rows, 256))).astype(np.float32)
    f[:, ::16] = 6.0
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, 0.1], np.float32)
    f[:50, 1:16] = ties[None]
    codes = torch.zeros((n_rows, 128), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((n_rows, 16), dtype=torch.uint8, device="cuda")
    dsv4.dsv4_quantize_fp4_rows(to_dev(f), n_rows, 256, codes, scales)
    assert (to_host(scales) == 0x38).all()
    g = to_host(codes)
    nib = np.stack([g & 0xF, g >> 4], axis=-1).reshape(n_rows, 256)
    assert np.array_equal(nib, O.e2m1_encode(f))


def test_pool_rows_matches_oracle():
    for ratio, dim in ((4, 128), (128, 512), (1, 64), (4, 128 + 8)):
        blocks = 300 if ratio < 128 else 40
        x = synth.bf16_bits(synth.normal(("pool", ratio, "x"), (blocks * ratio, dim)))
        z = synth.bf16_bits(synth.normal(("pool", ratio, "z"), (blocks * ratio, dim)))
        b = synth.normal(("pool", ratio, "b"), (ratio, dim), std=0.1)
        y = torch.zeros((blocks, dim), dtype=torch.float32, device="cuda")
        dsv4.dsv4_pool_rows(to_dev(x), to_dev(z), to_dev(b), blocks, ratio, dim, y)
        ref = O.pool_blocks(x, z, b, ratio)
        assert row_rel_err(to_host(y), ref).max() <= TOL
        assert row_rel_err(to_host(y), ref).max() <= 1e-5     # fp32 pooling is far inside the bar


# ----------------------------------------------------------------------------- append


@pytest.mark.parametrize("layer,n", [(W.CSA_4K, 4096), (W.HCA_128K, 131072)])
def test_append_builds_oracle_cache(layer, n):
    chunks = (4096,)
    desc, cache = gpu_stream_cache(layer, "append", 0, n, chunks)
    assert dsv4.dsv4_read_status(cache) == 0
    oc = oracle_stream_cache(layer, "append", 0, n, 0)
    n_c = n // layer.ratio
    assert to_host(cache.n_tokens)[0] == n
    dk = pooling_error_bound(oc, "k")
    compare_fp8_entries(to_host(cache.k_nope)[0, :n_c], to_host(cache.k_scale)[0, :n_c], oc["k_nope"], oc["k_scale"],
                        oc["pooled_k"], layer.d_nope, dk)
    compare_bf16(to_host(cache.k_rope, np.uint16)[0, :n_c], oc["k_rope"], oc["pooled_k"][:, layer.d_nope:],
                 dk[:, layer.d_nope:])
    if layer.separate_v:
        dv = pooling_error_bound(oc, "v")
        compare_fp8_entries(to_host(cache.v_nope)[0, :n_c], to_host(cache.v_scale)[0, :n_c], oc["v_nope"],
                            oc["v_scale"], oc["pooled_v"], layer.d_nope, dv)
        compare_bf16(to_host(cache.v_rope, np.uint16)[0, :n_c], oc["v_rope"], oc["pooled_v"][:, layer.d_nope:],
                     dv[:, layer.d_nope:])
    if layer.idx_dim:
        compare_fp4_rows(to_host(cache.idx_codes)[0, :n_c], to_host(cache.idx_scales)[0, :n_c], oc["idx_codes"],
                         oc["idx_scales"], oc["pooled_u"], pooling_error_bound(oc, "u"))
    ring = to_host(cache.win_k, np.uint16)[0]
    for slot, tok in oc["ring_slots"].items():
        assert np.array_equal(ring[slot], oc["tokens"]["k"][tok])


def test_append_rope_and_pooled_values_within_bar():
    layer = W.CSA_4K
    n = 1024
    desc, cache = gpu_stream_cache(layer, "pooled", 0, n, (1000, 24))
    oc = oracle_stream_cache(layer, "pooled", 0, n, 0)
    toks = oc["tokens"]
    y = torch.zeros((n // 4, layer.dim), dtype=torch.float32, device="cuda")
    dsv4.dsv4_pool_rows(to_dev(toks["k"]), to_dev(toks["z"]), to_dev(synth.position_bias("pooled", 0, layer, "b")),
                        n // 4, 4, layer.dim, y)
    assert row_rel_err(to_host(y), oc["pooled_k"]).max() <= TOL
    rope = O.bf16_decode(to_host(cache.k_rope, np.uint16)[0, : n // 4])
    assert row_rel_err(rope, oc["pooled_k"][:, layer.d_nope:]).max() <= 2.0 ** -8


@pytest.mark.parametrize("separate_v", [True, False], ids=["separate_v", "shared_kv"])
def test_append_chunk_invariance_bytes(separate_v):
    """Appending the same tokens in chunks of 4096, 1, 3 and 1000 gives byte-identical
    caches (pending planes compared on the slots of the open block only), with
    separate K and V and with them shared (the chunked pooling then runs in
    192-thread CTAs)."""
    n = 1102
    layer = W.scaled(W.CSA_4K, n_tokens=n, separate_v=separate_v)
    ref = gpu_stream_cache(layer, "chunks", 0, n, (4096,))[1]
    open_slots = n % layer.ratio
    for chunks in ((1,), (3,), (1000, 7), (5, 128, 2)):
        c = gpu_stream_cache(layer, "chunks", 0, n, chunks)[1]
        for name in ("k_nope", "k_scale", "k_rope", "v_nope", "v_scale", "v_rope", "idx_codes", "idx_scales",
                     "win_k", "win_v", "n_tokens"):
            if getattr(ref, name) is not None:
                assert torch.equal(getattr(ref, name), getattr(c, name)), (chunks, name)
        for name in ("pend_k", "pend_z", "pend_v", "pend_u", "pend_zu"):
            if getattr(ref, name) is not None:
                assert torch.equal(getattr(ref, name)[:, :open_slots], getattr(c, name)[:, :open_slots]), \
                    (chunks, name)


def test_append_capacity_overflow_sets_status_and_changes_nothing():
    layer = W.scaled(W.CSA_4K, n_tokens=64)
    desc, cache = gpu_stream_cache(layer, "cap", 0, 64, (64,), capacity=16)
    before = {n: getattr(cache, n).clone() for n in ("k_nope", "n_tokens", "win_k", "pend_k")}
    toks = {k: to_dev(v) for k, v in synth.token_stream("cap", 0, layer, 1, 64, 72).items()}
    b = to_dev(synth.position_bias("cap", 0, layer, "b"))
    bu = to_dev(synth.position_bias("cap", 0, layer, "bu"))
    dsv4.dsv4_compress_append(desc, cache, 8, toks["k"], toks["v"], toks["z"], b, toks["u"], toks["zu"], bu)
    assert dsv4.dsv4_read_status(cache) == dsv4.STATUS_CAPACITY
    for n_, t in before.items():
        assert torch.equal(t, getattr(cache, n_)), n_
    assert dsv4.dsv4_read_status(cache) == 0


# ----------------------------------------------------------------------------- indexer + top-k


def _index(desc, cache, layer, dec, k):
    B = layer.batch
    topk = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    scores = torch.zeros((B, desc.capacity), dtype=torch.float32, device="cuda")
    ws = dsv4.workspace(desc, max(layer.heads, 1), layer.idx_heads, k)
    dsv4.dsv4_index_topk(desc, cache, layer.idx_heads, to_dev(dec["q_idx"]), to_dev(dec["w"]), k, topk, scores, ws)
    torch.cuda.synchronize()
    return to_host(topk), to_host(scores)


def test_index_topk_csa_4k():
    layer = W.CSA_4K
    desc, cache = gpu_stream_cache(layer, "idx", 0, layer.n_tokens, (4096,))
    oc = oracle_stream_cache(layer, "idx", 0, layer.n_tokens, 0)
    dec = synth.decode_inputs("idx", 0, layer)
    g_topk, g_scores = _index(desc, cache, layer, dec, layer.topk)
    n_c = layer.n_comp
    o_scores = O.index_scores(oc["idx_codes"], oc["idx_scales"], dec["q_idx"][0], dec["w"][0])
    rel = np.abs(g_scores[0, :n_c] - o_scores) / np.maximum(np.abs(o_scores).max(), 1e-30)
    assert rel.max() <= 1e-5
    check_topk(g_topk[0], o_scores, O.topk_blocks(o_scores, layer.topk), layer.topk)


@pytest.mark.parametrize("n_c,k", [(0, 8), (5, 8), (8, 8), (300, 1), (2500, 2048)])
def test_index_topk_short_and_edge(n_c, k):
    layer = W.scaled(W.CSA_B32_128K, batch=2, n_tokens=n_c * 4, topk=k)
    planes = oracle_direct_planes(layer, "idxedge", n_c, range(2))
    desc, cache = gpu_cache_from_planes(layer, planes)
    dec = synth.decode_inputs("idxedge", n_c, layer)
    g_topk, g_scores = _index(desc, cache, layer, dec, k)
    for b in range(2):
        o_scores = O.index_scores(planes[b]["idx_codes"], planes[b]["idx_scales"], dec["q_idx"][b], dec["w"][b])
        check_topk(g_topk[b], o_scores, O.topk_blocks(o_scores, k), k)


@pytest.mark.parametrize("layer", [W.scaled(W.CSA_B32_128K, batch=2), W.scaled(W.STACK_CSA, batch=1)],
                         ids=["csa_b32_128k_shape", "stack_1m_shape"])
def test_index_topk_full_size_planted(layer):
    """Full-size selections with 1% planted keys: 32768 blocks (the planted keys
    are all selected and the boundary falls among random keys) and 2^18 blocks
    (2622 identical planted keys compete for 512 slots: the lowest indices win)."""
    planes = oracle_direct_planes(layer, "idxfull", 0, range(layer.batch))
    desc, cache = gpu_cache_from_planes(layer, planes)
    dec = synth.decode_inputs("idxfull", 0, layer)
    g_topk, g_scores = _index(desc, cache, layer, dec, layer.topk)
    for b in range(layer.batch):
        o_scores = O.index_scores(planes[b]["idx_codes"], planes[b]["idx_scales"], dec["q_idx"][b], dec["w"][b])
        rel = np.abs(g_scores[b, :layer.n_comp] - o_scores) / np.abs(o_scores).max()
        assert rel.max() <= 1e-5
        o_sel = O.topk_blocks(o_scores, layer.topk)
        check_topk(g_topk[b], o_scores, o_sel, layer.topk)
        planted = set(planes[b]["planted"].tolist())
        if len(planted) >= layer.topk:
            assert set(g_topk[b].tolist()) == set(sorted(planted)[:layer.topk])
        else:
            assert planted <= set(g_topk[b].tolist())
    # the attention over that selection (32-row tiles at batch 1 and 2)
    g_out, g_lse = _decode(desc, cache, layer, dec["q"], to_dev(g_topk), layer.topk)
    for b in range(layer.batch):
        o_out, o_lse = _oracle_attend_planes(layer, planes[b], dec["q"][b], g_topk[b])
        assert row_rel_err(g_out[b], o_out).max() <= TOL
        assert np.abs(g_lse[b] - o_lse).max() <= 1e-3


@pytest.mark.parametrize("n_c", [5000, 70000])
def test_topk_ties_go_to_lower_index(n_c):
    """All keys identical: every score ties, so the selection is the lowest k
    indices (at 70000 blocks more tied keys than a selecting CTA lists)."""
    layer = W.scaled(W.CSA_B32_128K, batch=1, n_tokens=4 * n_c, topk=512)
    desc = dsv4.layer_desc(layer, layer.capacity())
    cache = dsv4.Cache(desc)
    cache.idx_codes.fill_(0x23)
    cache.idx_scales.fill_(0x38)
    cache.n_tokens.fill_(layer.n_tokens)
    dec = synth.decode_inputs("ties", 0, layer)
    g_topk, g_scores = _index(desc, cache, layer, dec, 512)
    assert (g_topk[0] == np.arange(512)).all()


# ----------------------------------------------------------------------------- attention


def _decode(desc, cache, layer, q, topk=None, k=0):
    B, H = layer.batch, layer.heads
    out = torch.full((B, H, layer.dim), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = dsv4.workspace(desc, H, layer.idx_heads, max(k, layer.topk))
    if topk is None:
        dsv4.dsv4_hca_decode(desc, cache, H, to_dev(q), layer.sm_scale, out, lse, ws)
    else:
        dsv4.dsv4_csa_decode(desc, cache, H, to_dev(q), layer.sm_scale, topk, k, out, lse, ws)
    torch.cuda.synchronize()
    return to_host(out), to_host(lse)


def _oracle_attend_stream(layer, oc, q, sel):
    args = (oc["n_tokens"], layer.ratio, layer.window, oc["k_nope"], oc["k_scale"], oc["k_rope"], oc["ring_k"])
    if layer.separate_v:
        args += (oc["v_nope"], oc["v_scale"], oc["v_rope"], oc["ring_v"])
    if sel is None:
        return O.hca_attend(q, np.float32(layer.sm_scale), *args)
    return O.csa_attend(q, np.float32(layer.sm_scale), sel, *args)


def test_csa_decode_csa_4k_given_and_chained_topk():
    layer = W.CSA_4K
    desc, cache = gpu_stream_cache(layer, "csa", 0, layer.n_tokens, (4096,))
    oc = oracle_stream_cache(layer, "csa", 0, layer.n_tokens, 0)
    dec = synth.decode_inputs("csa", 0, layer)
    o_scores = O.index_scores(oc["idx_codes"], oc["idx_scales"], dec["q_idx"][0], dec["w"][0])
    o_sel = O.topk_blocks(o_scores, layer.topk)
    o_out, o_lse = _oracle_attend_stream(layer, oc, dec["q"][0], o_sel)
    # (1) the oracle's selection fed to the CUDA attention
    g_out, g_lse = _decode(desc, cache, layer, dec["q"], to_dev(o_sel[None]), layer.topk)
    assert row_rel_err(g_out[0], o_out).max() <= TOL
    assert np.abs(g_lse[0] - o_lse).max() <= 1e-3
    # (2) the CUDA chain index_topk -> csa_decode
    g_topk, _ = _index(desc, cache, layer, dec, layer.topk)
    check_topk(g_topk[0], o_scores, o_sel, layer.topk)
    g_out2, _ = _decode(desc, cache, layer, dec["q"], to_dev(g_topk), layer.topk)
    assert row_rel_err(g_out2[0], o_out).max() <= TOL


def test_hca_decode_hca_128k():
    layer = W.HCA_128K
    desc, cache = gpu_stream_cache(layer, "hca", 0, layer.n_tokens, (4096,))
    oc = oracle_stream_cache(layer, "hca", 0, layer.n_tokens, 0)
    dec = synth.decode_inputs("hca", 0, layer)
    o_out, o_lse = _oracle_attend_stream(layer, oc, dec["q"][0], None)
    g_out, g_lse = _decode(desc, cache, layer, dec["q"])
    assert row_rel_err(g_out[0], o_out).max() <= TOL
    assert np.abs(g_lse[0] - o_lse).max() <= 1e-3


def _oracle_attend_planes(layer, p, q, sel):
    args = (layer.n_tokens, layer.ratio, layer.window, p["k_nope"], p["k_scale"], p["k_rope"], p["ring_k"])
    if sel is None:
        return O.hca_attend(q, np.float32(layer.sm_scale), *args)
    return O.csa_attend(q, np.float32(layer.sm_scale), sel, *args)


@pytest.mark.parametrize("n_tokens,cap_extra", [(128 * 1000 + 77, None), (128 * 257, None), (128 * 40 + 5, None),
                                                (128 * 257 + 9, 2)])
def test_hca_decode_stack_shape(n_tokens, cap_extra):
    """D = 512 (448 FP8 + 64 RoPE), 64 heads, K = V, four sequences as in the
    decode step: compressed rows by TMA boxes over several tiles per CTA, a
    partial last tile, the window tile; small contexts take 64- and 32-row
    tiles. A capacity that is not a multiple of 4 takes the scales by loads
    instead of bulk copies."""
    layer = W.scaled(W.STACK_HCA, n_tokens=n_tokens)
    planes = oracle_direct_planes(layer, "hcastack", 1, range(layer.batch))
    cap = None if cap_extra is None else layer.n_comp + cap_extra
    desc, cache = gpu_cache_from_planes(layer, planes, capacity=cap)
    dec = synth.decode_inputs("hcastack", 1, layer)
    g_out, g_lse = _decode(desc, cache, layer, dec["q"])
    assert dsv4.dsv4_read_status(cache) == 0
    for b in range(layer.batch):
        o_out, o_lse = _oracle_attend_planes(layer, planes[b], dec["q"][b], None)
        assert row_rel_err(g_out[b], o_out).max() <= TOL
        assert np.abs(g_lse[b] - o_lse).max() <= 1e-3


def test_hca_decode_full_size_decode_step():
    """The decode step's HCA layer at full size (the benchmark's launch):
    four sequences of 2^20 tokens, 8192 compressed entries each."""
    layer = W.STACK_HCA
    planes = oracle_direct_planes(layer, "hcafull", 1, range(layer.batch), processes=4)
    desc, cache = gpu_cache_from_planes(layer, planes, extra=64)
    dec = synth.decode_inputs("hcafull", 1, layer)
    g_out, g_lse = _decode(desc, cache, layer, dec["q"])
    assert dsv4.dsv4_read_status(cache) == 0
    for b in range(layer.batch):
        o_out, o_lse = _oracle_attend_planes(layer, planes[b], dec["q"][b], None)
        assert row_rel_err(g_out[b], o_out).max() <= TOL
        assert np.abs(g_lse[b] - o_lse).max() <= 1e-3


@pytest.mark.parametrize("n_tokens", [4 * 3000 + 3, 4 * 400])
def test_csa_decode_stack_shape_chained(n_tokens):
    """D = 512 CSA with four sequences (tiles of 32 rows): index_topk ->
    csa_decode; the selection is checked against the oracle's, the attention
    against the oracle's attention over the same selection."""
    layer = W.scaled(W.STACK_CSA, n_tokens=n_tokens)
    planes = oracle_direct_planes(layer, "csastack", 0, range(layer.batch))
    desc, cache = gpu_cache_from_planes(layer, planes)
    dec = synth.decode_inputs("csastack", 0, layer)
    g_topk, _ = _index(desc, cache, layer, dec, layer.topk)
    g_out, g_lse = _decode(desc, cache, layer, dec["q"], to_dev(g_topk), layer.topk)
    assert dsv4.dsv4_read_status(cache) == 0
    for b in range(layer.batch):
        o_scores = O.index_scores(planes[b]["idx_codes"], planes[b]["idx_scales"], dec["q_idx"][b], dec["w"][b])
        check_topk(g_topk[b], o_scores, O.topk_blocks(o_scores, layer.topk), layer.topk)
        o_out, o_lse = _oracle_attend_planes(layer, planes[b], dec["q"][b], g_topk[b])
        assert row_rel_err(g_out[b], o_out).max() <= TOL
        assert np.abs(g_lse[b] - o_lse).max() <= 1e-3


@pytest.mark.parametrize("n", [0, 1, 3, 4, 5, 127, 128, 129, 700])
def test_short_contexts(n):
    """Empty cache, fewer tokens than the window, fewer blocks than k."""
    layer = W.scaled(W.CSA_4K, n_tokens=n)
    desc, cache = gpu_stream_cache(layer, "short", n, n, (max(n, 1),), capacity=max(1, n // 4 + 1))
    oc = oracle_stream_cache(layer, "short", n, n, 0)
    dec = synth.decode_inputs("short", n, layer)
    g_topk, g_scores = _index(desc, cache, layer, dec, layer.topk)
    n_c = n // 4
    if n_c:
        o_scores = O.index_scores(oc["idx_codes"], oc["idx_scales"], dec["q_idx"][0], dec["w"][0])
    else:
        o_scores = np.zeros(0)
    o_sel = O.topk_blocks(o_scores, layer.topk)
    assert np.array_equal(g_topk[0], o_sel)          # n_c <= k: all blocks then -1
    g_out, g_lse = _decode(desc, cache, layer, dec["q"], to_dev(g_topk), layer.topk)
    o_out, o_lse = _oracle_attend_stream(layer, oc, dec["q"][0], o_sel)
    if n == 0:
        assert (g_out == 0).all() and np.isneginf(g_lse).all()
    else:
        assert row_rel_err(g_out[0], o_out).max() <= TOL
    gh, _ = _decode(desc, cache, W.scaled(layer, kind="hca"), dec["q"])
    oh, _ = _oracle_attend_stream(layer, oc, dec["q"][0], None)
    if n:
        assert row_rel_err(gh[0], oh).max() <= TOL


def test_ratio1_all_selected_no_window_is_full_attention():
    """CSA with ratio 1, top-k = every entry and no window is full softmax
    attention over the dequantised cache (checked against torch SDPA, fp64)."""
    layer = W.Layer("csa", 2, 200, 8, 64, 64, False, 1, 0, idx_heads=4, idx_dim=64, topk=200,
                    cache_source="direct")
    planes = oracle_direct_planes(layer, "full", 0, range(2))
    desc, cache = gpu_cache_from_planes(layer, planes)
    dec = synth.decode_inputs("full", 0, layer)
    sel = np.tile(np.arange(200, dtype=np.int32), (2, 1))
    g_out, _ = _decode(desc, cache, layer, dec["q"], to_dev(sel), 200)
    for b in range(2):
        K = O.dequant_kv_rows(planes[b]["k_nope"], planes[b]["k_scale"], planes[b]["k_rope"])
        qt = torch.from_numpy(O.bf16_decode(dec["q"][b]))[None, :, None, :]
        kt = torch.from_numpy(K)[None, None].expand(1, 8, 200, 128)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, kt, scale=float(np.float32(layer.sm_scale)))
        assert row_rel_err(g_out[b], ref[0, :, 0].numpy()).max() <= TOL


def test_bad_topk_index_sets_status_and_is_ignored():
    layer = W.scaled(W.CSA_B32_128K, batch=1, n_tokens=4 * 100, topk=4)
    planes = oracle_direct_planes(layer, "bad", 0, [0])
    desc, cache = gpu_cache_from_planes(layer, planes)
    dec = synth.decode_inputs("bad", 0, layer)
    sel = np.array([[3, 100, -5, 7]], np.int32)
    g_out, _ = _decode(desc, cache, layer, dec["q"], to_dev(sel), 4)
    assert dsv4.dsv4_read_status(cache) == dsv4.STATUS_BAD_INDEX
    p = planes[0]
    o_out, _ = O.csa_attend(dec["q"][0], np.float32(layer.sm_scale), np.array([3, 7]), layer.n_tokens, 4, 128,
                            p["k_nope"], p["k_scale"], p["k_rope"], p["ring_k"])
    assert row_rel_err(g_out[0], o_out).max() <= TOL


def test_host_validation_errors_launch_nothing():
    layer = W.CSA_4K
    desc = dsv4.layer_desc(layer, 100)
    cache = dsv4.Cache(desc)
    ws = dsv4.workspace(desc, 16, 4, 64)
    q = torch.zeros((1, 16, 128), dtype=torch.int16, device="cuda")
    out = torch.zeros((1, 16, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(dsv4.Dsv4Error) as e:
        dsv4.dsv4_hca_decode(desc, cache, 0, q, 0.1, out, None, ws)
    assert e.value.code == dsv4.ERR_INVALID_ARG
    with pytest.raises(dsv4.Dsv4Error) as e:
        dsv4.dsv4_hca_decode(desc, cache, 16, q, 0.1, out, None, ws[:100])
    assert e.value.code == dsv4.ERR_WORKSPACE
    with pytest.raises(dsv4.Dsv4Error) as e:
        dsv4.dsv4_hca_decode(desc, cache, 16, q.view(-1)[1:], 0.1, out, None, ws)
    assert e.value.code == dsv4.ERR_MISALIGNED
    bad = dsv4.LayerDesc(1, 60, 64, 4, 128, 1, 64, 100)
    with pytest.raises(dsv4.Dsv4Error) as e:
        dsv4.dsv4_hca_decode(bad, cache, 16, q, 0.1, out, None, ws)
    assert e.value.code == dsv4.ERR_UNSUPPORTED
