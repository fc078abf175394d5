"""GPU parity at the shapes the benchmark and the declared limits reach, and at
the layer variants beyond the decode step: the batched CSA configuration at
B = 32 (128-row gathered tiles, two per CTA), the compressor at D = 512 with
128-dim FP4 indexer keys (ratio 4 and 128, chunked and single-token appends,
pending planes), the CUDA-core attention path, 256-dim indexer keys, 128
query and indexer heads, entries and window tokens far from unit magnitude,
the window-only layer (k = 0), the ratio-1 selection on raw tokens, and a
cache copied out to the host and back between appends.

Every expected value comes from the float64 oracle on the same seeded inputs
(the oracle quantises the planes uploaded to the device). Bars as in
test_gpu_parity: quantised bytes bit-exact except at the stated rounding and
tie exceptions, attention within 2e-3 max relative error per row."""
import numpy as np
import pytest
import torch

import oracle as O
from compressed_sparse_kv_05_b300 import dsv4, synth
from compressed_sparse_kv_05_b300 import workloads as W

from .gpu_util import (check_pending, check_topk, compare_bf16, compare_fp4_rows, compare_fp8_entries,
                       gpu_cache_from_planes, gpu_stream_cache, oracle_attend_planes, oracle_direct_planes,
                       oracle_stream_cache, planes_from_rows, pooling_error_bound, row_rel_err, to_dev, to_host)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

TOL = 2e-3


def _index(desc, cache, layer, dec, k):
    B = layer.batch
    topk = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    scores = torch.zeros((B, desc.capacity), dtype=torch.float32, device="cuda")
    ws = dsv4.workspace(desc, max(layer.heads, 1), layer.idx_heads, k)
    dsv4.dsv4_index_topk(desc, cache, layer.idx_heads, to_dev(dec["q_idx"]), to_dev(dec["w"]), k, topk, scores, ws)
    torch.cuda.synchronize()
    return to_host(topk), to_host(scores)


def _decode(desc, cache, layer, q, topk=None, k=0, hca=False):
    B, H = layer.batch, layer.heads
    out = torch.full((B, H, layer.dim), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = dsv4.workspace(desc, H, layer.idx_heads, max(k, layer.topk))
    if hca:
        dsv4.dsv4_hca_decode(desc, cache, H, to_dev(q), layer.sm_scale, out, lse, ws)
    else:
        dsv4.dsv4_csa_decode(desc, cache, H, to_dev(q), layer.sm_scale, topk, k, out, lse, ws)
    torch.cuda.synchronize()
    return to_host(out), to_host(lse)


def _check_attention(g_out, g_lse, o_out, o_lse):
    assert np.isfinite(g_out).all()
    assert row_rel_err(g_out, o_out).max() <= TOL
    assert np.abs(g_lse - o_lse).max() <= 1e-3


def _check_chain(layer, planes, desc, cache, dec, g_topk):
    """The GPU's selection against the oracle's (set parity with the tie
    exception); then attention: over the oracle's own selection (uploaded) for
    every sequence, and the chained call over the GPU's selection wherever the
    two selections agree, both against the oracle's attention over its own
    selection. Returns the oracle's selections."""
    o_sel = []
    for b in range(layer.batch):
        o_scores = O.index_scores(planes[b]["idx_codes"], planes[b]["idx_scales"], dec["q_idx"][b], dec["w"][b])
        o_sel.append(O.topk_blocks(o_scores, layer.topk))
        check_topk(g_topk[b], o_scores, o_sel[b], layer.topk)
    o_sel = np.stack(o_sel)
    c_out, c_lse = _decode(desc, cache, layer, dec["q"], to_dev(g_topk), layer.topk)
    g_out, g_lse = _decode(desc, cache, layer, dec["q"], to_dev(o_sel), layer.topk)
    assert dsv4.dsv4_read_status(cache) == 0
    agree = 0
    for b in range(layer.batch):
        o_out, o_lse = oracle_attend_planes(layer, planes[b], dec["q"][b], o_sel[b])
        _check_attention(g_out[b], g_lse[b], o_out, o_lse)
        if np.array_equal(g_topk[b], o_sel[b]):
            agree += 1
            _check_attention(c_out[b], c_lse[b], o_out, o_lse)
    print(f"chained selection identical to the oracle's in {agree} of {layer.batch} sequences")
    return o_sel


# ----------------------------------------------------------------------------- batched CSA (B = 32)


def test_csa_batch32_plan_small_context():
    """B = 32 with a short context reaches the plan of the batched configuration
    (128-row gathered tiles, two per CTA, three splits a sequence): the chain
    index_topk -> csa_decode against the oracle."""
    layer = W.scaled(W.CSA_B32_128K, n_tokens=4 * 2000 + 3)
    desc = dsv4.layer_desc(layer, layer.capacity())
    plan = dsv4.dsv4_decode_plan(desc, layer.heads, layer.topk)
    assert plan["tile_rows"] == 128 and plan["tiles_per_split"] == 2, plan
    planes = oracle_direct_planes(layer, "b32small", 0, range(layer.batch), processes=8)
    desc, cache = gpu_cache_from_planes(layer, planes)
    dec = synth.decode_inputs("b32small", 0, layer)
    g_topk, _ = _index(desc, cache, layer, dec, layer.topk)
    _check_chain(layer, planes, desc, cache, dec, g_topk)


def test_csa_batch32_full_size():
    """The batched CSA configuration at full size: 32 sequences of 32768
    compressed entries (1% planted keys), top-512, window 128, 64 heads over a
    shared 512-dim entry, in the benchmark's launch configuration."""
    layer = W.CSA_B32_128K
    planes = oracle_direct_planes(layer, "b32full", 0, range(layer.batch), processes=8)
    desc, cache = gpu_cache_from_planes(layer, planes, extra=64)
    plan = dsv4.dsv4_decode_plan(desc, layer.heads, layer.topk)
    assert plan["tile_rows"] == 128 and plan["tiles_per_split"] == 2, plan
    dec = synth.decode_inputs("b32full", 0, layer)
    g_topk, g_scores = _index(desc, cache, layer, dec, layer.topk)
    for b in range(layer.batch):
        o_scores = O.index_scores(planes[b]["idx_codes"], planes[b]["idx_scales"], dec["q_idx"][b], dec["w"][b])
        assert (np.abs(g_scores[b, :layer.n_comp] - o_scores) / np.abs(o_scores).max()).max() <= 1e-5
        assert set(planes[b]["planted"].tolist()) <= set(g_topk[b].tolist())
    _check_chain(layer, planes, desc, cache, dec, g_topk)


# ----------------------------------------------------------------------------- compressor at D = 512


def _check_stream_cache(layer, cache, n, tag):
    n_c = n // layer.ratio
    assert (to_host(cache.n_tokens) == n).all()
    for b in range(layer.batch):
        oc = oracle_stream_cache(layer, tag, 0, n, b)
        dk = pooling_error_bound(oc, "k")
        compare_fp8_entries(to_host(cache.k_nope)[b, :n_c], to_host(cache.k_scale)[b, :n_c], oc["k_nope"],
                            oc["k_scale"], oc["pooled_k"], layer.d_nope, dk)
        compare_bf16(to_host(cache.k_rope, np.uint16)[b, :n_c], oc["k_rope"], oc["pooled_k"][:, layer.d_nope:],
                     dk[:, layer.d_nope:])
        if layer.idx_dim:
            compare_fp4_rows(to_host(cache.idx_codes)[b, :n_c], to_host(cache.idx_scales)[b, :n_c], oc["idx_codes"],
                             oc["idx_scales"], oc["pooled_u"], pooling_error_bound(oc, "u"))
        ring = to_host(cache.win_k, np.uint16)[b]
        for slot, tok in oc["ring_slots"].items():
            assert np.array_equal(ring[slot], oc["tokens"]["k"][tok])
        check_pending(cache, oc, layer, b)


@pytest.mark.parametrize("base", [W.STACK_CSA, W.STACK_HCA], ids=["ratio4_idx128", "ratio128"])
def test_append_d512_chunked(base):
    """4096-token chunks (the compressor configuration's chunking) into a
    448 + 64 cache, with 128-dim FP4 indexer keys for ratio 4: entries, keys,
    window ring and the open block's pending tokens against the oracle."""
    n = 4096 * 3 + 77
    layer = W.scaled(base, batch=2, n_tokens=n, cache_source="stream")
    desc, cache = gpu_stream_cache(layer, "app512", 0, n, (4096,))
    assert dsv4.dsv4_read_status(cache) == 0
    _check_stream_cache(layer, cache, n, "app512")


@pytest.mark.parametrize("base", [W.STACK_CSA, W.STACK_HCA], ids=["ratio4_idx128", "ratio128"])
def test_append_d512_single_tokens(base):
    """The decode step's single-token appends at D = 512 (the kernel the
    benchmark runs): a 4096-token prefix, then 300 appends of one token, which
    complete 75 ratio-4 blocks or 2 ratio-128 blocks through the pending planes."""
    n = 4096 + 300
    layer = W.scaled(base, batch=2, n_tokens=n, cache_source="stream")
    desc, cache = gpu_stream_cache(layer, "app512t1", 0, n, (4096,) + (1,) * 300)
    assert dsv4.dsv4_read_status(cache) == 0
    _check_stream_cache(layer, cache, n, "app512t1")


@pytest.mark.parametrize("base", [W.HCA_128K, W.STACK_HCA], ids=["d128_sep_v", "d512"])
def test_long_block_chunk_invariance_bytes(base):
    """Ratio-128 layers pool a chunk's blocks with each block's channels split
    over a cluster of CTAs, single tokens with one CTA: the caches are
    byte-identical whatever the chunking (blocks straddling two calls
    included), for a separate-V 128-dim layer (clusters of 2) and the 448 + 64
    layer (clusters of 8)."""
    n = 128 * 5 + 37
    layer = W.scaled(base, batch=2, n_tokens=n, cache_source="stream")
    ref = gpu_stream_cache(layer, "lbchunks", 0, n, (4096,))[1]
    open_slots = n % layer.ratio
    for chunks in ((1,), (300, 7), (5, 128, 2), (200,)):
        c = gpu_stream_cache(layer, "lbchunks", 0, n, chunks)[1]
        assert dsv4.dsv4_read_status(c) == 0
        for name in ("k_nope", "k_scale", "k_rope", "v_nope", "v_scale", "v_rope", "win_k", "win_v", "n_tokens"):
            if getattr(ref, name) is not None:
                assert torch.equal(getattr(ref, name), getattr(c, name)), (chunks, name)
        for name in ("pend_k", "pend_z", "pend_v"):
            if getattr(ref, name) is not None:
                assert torch.equal(getattr(ref, name)[:, :open_slots], getattr(c, name)[:, :open_slots]), (chunks, name)


@pytest.mark.parametrize("ratio,sep,d_nope", [(16, True, 64), (256, False, 64), (128, False, 128), (64, True, 256)],
                         ids=["ratio16_sep_v", "ratio256", "d192_cs3", "d320_cs5_sep_v"])
def test_long_block_other_token_groups(ratio, sep, d_nope):
    """The clustered pooling at its other team shapes: 2 token groups at ratio
    16 (2 channels a thread, separate V) and 32 at ratio 256 (8 channels a
    thread) with 128-dim entries (clusters of 2), and clusters of 3 and 5 CTAs
    (192- and 320-dim entries): chunked appends whose blocks straddle calls
    against the oracle, and byte-identical to single-token appends."""
    n = ratio * 6 + 5
    layer = W.Layer("hca", 2, n, 8, d_nope, 64, sep, ratio, 128)
    desc, cache = gpu_stream_cache(layer, "lbgroups", 0, n, (2 * ratio + 3,))
    assert dsv4.dsv4_read_status(cache) == 0
    _check_stream_cache(layer, cache, n, "lbgroups")
    one = gpu_stream_cache(layer, "lbgroups", 0, n, (1,))[1]
    for name in ("k_nope", "k_scale", "k_rope", "v_nope", "v_scale", "v_rope", "win_k", "win_v", "n_tokens"):
        if getattr(cache, name) is not None:
            assert torch.equal(getattr(cache, name), getattr(one, name)), name


def test_long_block_capacity_overflow_sets_status_and_changes_nothing():
    """A chunk that would complete more ratio-128 blocks than the cache holds
    (the clustered path) sets the capacity bit and writes nothing."""
    layer = W.scaled(W.STACK_HCA, batch=2, n_tokens=256, cache_source="stream")
    desc, cache = gpu_stream_cache(layer, "lbcap", 0, 256, (256,), capacity=3)
    assert dsv4.dsv4_read_status(cache) == 0
    before = {n: getattr(cache, n).clone() for n in ("k_nope", "k_scale", "k_rope", "n_tokens", "win_k", "pend_k")}
    toks = {k: to_dev(v) for k, v in synth.token_stream("lbcap", 0, layer, 2, 256, 512).items()}
    b = to_dev(synth.position_bias("lbcap", 0, layer, "b"))
    dsv4.dsv4_compress_append(desc, cache, 256, toks["k"], None, toks["z"], b)
    assert dsv4.dsv4_read_status(cache) == dsv4.STATUS_CAPACITY
    for n_, t in before.items():
        assert torch.equal(t, getattr(cache, n_)), n_
    assert dsv4.dsv4_read_status(cache) == 0


# ----------------------------------------------------------------------------- other declared shapes


@pytest.mark.parametrize("d_nope,d_rope,sep", [(128, 64, False), (256, 64, True)], ids=["d192_shared", "d320_sep"])
def test_cuda_core_attention_path(d_nope, d_rope, sep):
    """Shapes the tensor-core kernel does not take (D not a multiple of 128, or
    separate V beyond 256 dims) run the CUDA-core split kernel and its merge."""
    layer = W.Layer("csa", 2, 4 * 700 + 1, 24, d_nope, d_rope, sep, 4, 128, idx_heads=8, idx_dim=64, topk=96,
                    cache_source="direct", planted_frac=0.01)
    desc = dsv4.layer_desc(layer, layer.capacity())
    assert dsv4.dsv4_decode_plan(desc, layer.heads, layer.topk)["tensor_core"] == 0
    planes = oracle_direct_planes(layer, "cudacore", 0, range(layer.batch))
    desc, cache = gpu_cache_from_planes(layer, planes)
    dec = synth.decode_inputs("cudacore", 0, layer)
    g_topk, _ = _index(desc, cache, layer, dec, layer.topk)
    _check_chain(layer, planes, desc, cache, dec, g_topk)
    h_out, h_lse = _decode(desc, cache, layer, dec["q"], hca=True)
    for b in range(layer.batch):
        _check_attention(h_out[b], h_lse[b], *oracle_attend_planes(layer, planes[b], dec["q"][b], None))


def test_indexer_keys_256_dims():
    """idx_dim = 256 (the widest declared indexer key): scores and selection."""
    layer = W.Layer("csa", 2, 4 * 5000, 64, 448, 64, False, 4, 128, idx_heads=64, idx_dim=256, topk=128,
                    cache_source="direct", planted_frac=0.01)
    planes = oracle_direct_planes(layer, "idx256", 0, range(layer.batch))
    desc, cache = gpu_cache_from_planes(layer, planes)
    dec = synth.decode_inputs("idx256", 0, layer)
    g_topk, g_scores = _index(desc, cache, layer, dec, layer.topk)
    for b in range(layer.batch):
        o_scores = O.index_scores(planes[b]["idx_codes"], planes[b]["idx_scales"], dec["q_idx"][b], dec["w"][b])
        assert (np.abs(g_scores[b, :layer.n_comp] - o_scores) / np.abs(o_scores).max()).max() <= 1e-5
        check_topk(g_topk[b], o_scores, O.topk_blocks(o_scores, layer.topk), layer.topk)


def test_128_query_and_indexer_heads():
    """H = 128 (two head groups of 64 per sequence) and Hi = 128 (the padded
    indexer width 128): the chain and the HCA call against the oracle."""
    layer = W.Layer("csa", 2, 4 * 3000 + 2, 128, 448, 64, False, 4, 128, idx_heads=128, idx_dim=128, topk=256,
                    cache_source="direct", planted_frac=0.01)
    assert dsv4.dsv4_decode_plan(dsv4.layer_desc(layer, layer.capacity()), 128, 256)["head_groups"] == 2
    planes = oracle_direct_planes(layer, "h128", 0, range(layer.batch))
    desc, cache = gpu_cache_from_planes(layer, planes)
    dec = synth.decode_inputs("h128", 0, layer)
    g_topk, _ = _index(desc, cache, layer, dec, layer.topk)
    _check_chain(layer, planes, desc, cache, dec, g_topk)
    h_out, h_lse = _decode(desc, cache, layer, dec["q"], hca=True)
    for b in range(layer.batch):
        _check_attention(h_out[b], h_lse[b], *oracle_attend_planes(layer, planes[b], dec["q"][b], None))


# ----------------------------------------------------------------------------- magnitudes far from 1


def _wide_planes(layer, tag):
    """Four sequences whose entries and window tokens sit far from unit
    magnitude: (0) all entries and the window scaled by 2^-20; (1) all by 2^10;
    (2) each entry by its own 2^u, u ~ U(-20, 10), with a window of 2^-20;
    (3) unit entries with a window scaled by 2^12."""
    r = np.random.default_rng(synth._parts((tag,))[0])
    n_c, W_, D = layer.n_comp, min(layer.window, layer.n_tokens), layer.dim
    planes = []
    for b in range(layer.batch):
        kv = synth.normal((tag, b, "kv"), (n_c, D))
        win = synth.normal((tag, b, "win"), (W_, D))
        if b == 0:
            kv, win = kv * 2.0 ** -20, win * 2.0 ** -20
        elif b == 1:
            kv, win = kv * 2.0 ** 10, win * 2.0 ** 10
        elif b == 2:
            kv, win = kv * np.exp2(r.uniform(-20, 10, (n_c, 1))), win * 2.0 ** -20
        else:
            win = win * 2.0 ** 12
        planes.append(planes_from_rows(layer, kv.astype(np.float32), synth.bf16_bits(win)))
    return planes


@pytest.mark.parametrize("kind", ["hca", "csa"])
def test_attention_far_from_unit_magnitude(kind):
    """Entry scales from 2^-27 to 2^9 and window tokens from 2^-20 to 2^14:
    every row of the output within the 2e-3 bar, and no RANGE status (no value
    reaches the f16 limit of 65504)."""
    base = W.STACK_HCA if kind == "hca" else W.STACK_CSA
    layer = W.scaled(base, n_tokens=base.ratio * 1500 + 1, cache_source="direct", planted_frac=0.0)
    planes = _wide_planes(layer, f"wide{kind}")
    desc, cache = gpu_cache_from_planes(layer, planes)
    q = synth.decode_inputs(f"wide{kind}", 0, layer)["q"]
    if kind == "hca":
        g_out, g_lse = _decode(desc, cache, layer, q, hca=True)
        sels = [None] * layer.batch
    else:
        sels = [np.sort(np.random.default_rng(b).choice(layer.n_comp, layer.topk, replace=False)).astype(np.int32)
                for b in range(layer.batch)]
        g_out, g_lse = _decode(desc, cache, layer, q, to_dev(np.stack(sels)), layer.topk)
    assert dsv4.dsv4_read_status(cache) == 0
    for b in range(layer.batch):
        o_out, o_lse = oracle_attend_planes(layer, planes[b], q[b], sels[b])
        assert row_rel_err(g_out[b], o_out).max() <= TOL, (b, row_rel_err(g_out[b], o_out).max())
        # The log-sum-exp inherits the scores' rounding: the f16 key operands carry
        # 11 significant bits, so a score moves by about 2^-11 of the size of its
        # terms (sm_scale * ||q (.) k||, large here: keys of 2^10 give scores near
        # 3000); 1e-3 absolute where the scores are of order one.
        p = planes[b]
        K = O.dequant_kv_rows(p["k_nope"], p["k_scale"], p["k_rope"])
        sel = np.arange(layer.n_comp) if sels[b] is None else sels[b]
        Kall = np.concatenate([K[sel], O.bf16_decode(p["ring_k"])], axis=0)
        qd = O.bf16_decode(q[b])
        size = layer.sm_scale * np.sqrt((qd ** 2) @ (Kall ** 2).T).max(axis=1)
        assert (np.abs(g_lse[b] - o_lse) <= 1e-3 + 2.0 ** -8 * size).all()


# ----------------------------------------------------------------------------- layer variants


def test_window_only_layer():
    """k = 0: attention over the sliding window alone (the standard window
    layer after the CSA / HCA stack), with the compressed entries ignored; also
    a context shorter than the window."""
    for n in (1500, 77):
        layer = W.scaled(W.CSA_4K, n_tokens=n)
        desc, cache = gpu_stream_cache(layer, "swa", n, n, (4096,))
        oc = oracle_stream_cache(layer, "swa", n, n, 0)
        q = synth.decode_inputs("swa", n, layer)["q"]
        g_out, g_lse = _decode(desc, cache, layer, q, None, 0)
        args = (n, layer.ratio, layer.window, oc["k_nope"], oc["k_scale"], oc["k_rope"], oc["ring_k"],
                oc["v_nope"], oc["v_scale"], oc["v_rope"], oc["ring_v"])
        o_out, o_lse = O.csa_attend(q[0], np.float32(layer.sm_scale), np.zeros(0, np.int32), *args)
        _check_attention(g_out[0], g_lse[0], o_out, o_lse)


def test_ratio1_selection_on_raw_tokens():
    """Ratio 1: every token is its own entry and the indexer selects among raw
    tokens (the selection space of the earlier sparse-attention design the
    pages contrast CSA with); appended, indexed and attended against the oracle."""
    n = 3000
    layer = W.Layer("csa", 2, n, 16, 64, 64, True, 1, 128, idx_heads=4, idx_dim=64, topk=256)
    desc, cache = gpu_stream_cache(layer, "ratio1", 0, n, (1000, 1, 999))
    assert dsv4.dsv4_read_status(cache) == 0
    dec = synth.decode_inputs("ratio1", 0, layer)
    g_topk, g_scores = _index(desc, cache, layer, dec, layer.topk)
    planes = []
    for b in range(layer.batch):
        oc = oracle_stream_cache(layer, "ratio1", 0, n, b)
        assert oc["idx_codes"].shape[0] == n and not oc["pending"]
        planes.append(oc)
    _check_chain(layer, planes, desc, cache, dec, g_topk)


def test_topk_beyond_one_cluster():
    """More blocks than one cluster of CTAs holds (ratio 1 over 600000 raw
    tokens, above 16 x 72 x 512): the selection takes the global-atomic kernel;
    with identical planted keys competing for the k slots, the lowest indices win."""
    n = 600000
    layer = W.Layer("csa", 1, n, 16, 64, 64, True, 1, 128, idx_heads=4, idx_dim=64, topk=512, planted_frac=0.002)
    planes = oracle_direct_planes(layer, "idxbig", 0, range(layer.batch))
    desc, cache = gpu_cache_from_planes(layer, planes)
    dec = synth.decode_inputs("idxbig", 0, layer)
    g_topk, g_scores = _index(desc, cache, layer, dec, layer.topk)
    o_scores = O.index_scores(planes[0]["idx_codes"], planes[0]["idx_scales"], dec["q_idx"][0], dec["w"][0])
    assert np.abs(g_scores[0, :n] - o_scores).max() / np.abs(o_scores).max() <= 1e-5
    o_sel = O.topk_blocks(o_scores, layer.topk)
    check_topk(g_topk[0], o_scores, o_sel, layer.topk)
    planted = sorted(planes[0]["planted"].tolist())
    assert len(planted) >= layer.topk and set(g_topk[0].tolist()) == set(planted[:layer.topk])


# ----------------------------------------------------------------------------- cache state round trip


def test_cache_round_trip_through_host():
    """The cache is the whole decode state: copied to host memory, restored into
    fresh device planes and appended to further, it gives the same bytes as a
    cache appended to without interruption."""
    n1, n2 = 1001, 523
    layer = W.scaled(W.CSA_4K, batch=2, n_tokens=n1 + n2)
    cap = (n1 + n2) // layer.ratio + 1
    desc, ref = gpu_stream_cache(layer, "trip", 0, n1, (1001,), capacity=cap)
    saved = {k: v.cpu() for k, v in vars(ref).items() if isinstance(v, torch.Tensor)}
    restored = dsv4.Cache(desc)
    for k, v in saved.items():
        getattr(restored, k).copy_(v)
    b = to_dev(synth.position_bias("trip", 0, layer, "b"))
    bu = to_dev(synth.position_bias("trip", 0, layer, "bu"))
    toks = {k: to_dev(v) for k, v in synth.token_stream("trip", 0, layer, layer.batch, n1, n1 + n2).items()}
    for c in (ref, restored):
        for t0, t1 in ((0, 200), (200, 201), (201, n2)):
            sl = {k: v[:, t0:t1].contiguous() for k, v in toks.items()}
            dsv4.dsv4_compress_append(desc, c, t1 - t0, sl["k"], sl["v"], sl["z"], b, sl["u"], sl["zu"], bu)
    torch.cuda.synchronize()
    for name, t in vars(ref).items():
        if isinstance(t, torch.Tensor):
            assert torch.equal(t, getattr(restored, name)), name
    # and the restored cache matches the oracle's cache of the whole stream
    oc = oracle_stream_cache(layer, "trip", 0, n1 + n2, 1)
    n_c = (n1 + n2) // layer.ratio
    compare_fp8_entries(to_host(restored.k_nope)[1, :n_c], to_host(restored.k_scale)[1, :n_c], oc["k_nope"],
                        oc["k_scale"], oc["pooled_k"], layer.d_nope, pooling_error_bound(oc, "k"))
    check_pending(restored, oc, layer, 1)
