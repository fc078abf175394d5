"""GPU parity of multi-token decode (T queries per sequence in one call, after
their tokens were appended): causal indexer scores and top-k per query, CSA
attention over each query's selection and window, HCA attention over the
entries complete at each query's position, against the float64 oracle on the
same seeded inputs; and T = 1 against the single-token calls."""
import numpy as np
import pytest
import torch

import oracle as O
from compressed_sparse_kv_05_b300 import dsv4, synth
from compressed_sparse_kv_05_b300 import workloads as W

from .gpu_util import (check_topk, gpu_cache_from_planes, gpu_stream_cache, oracle_direct_planes,
                       oracle_stream_cache, row_rel_err, to_dev, to_host)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

TOL = 2e-3


def _span(rows_bits, n, T, Wn):
    """Raw rows of the positions n - T - W + 1 .. n - 1 (zeros for negative positions)."""
    first = n - T - Wn + 1
    out = np.zeros((T + Wn - 1, rows_bits.shape[1]), np.uint16)
    lo = max(0, -first)
    out[lo:] = rows_bits[first + lo: n]
    return out


def _queries(tag, layer, T):
    """Queries of a step: q [B][T][H][D], q_idx [B][T][Hi][Di] bf16, w [B][T][Hi] ~U(0,1)."""
    B, H, D = layer.batch, layer.heads, layer.dim
    q = synth.bf16_bits(synth.normal(tag + ("q",), (B, T, H, D)))
    qi = synth.bf16_bits(synth.normal(tag + ("q_idx",), (B, T, layer.idx_heads, layer.idx_dim)))
    w = synth.uniform(tag + ("w",), (B, T, layer.idx_heads))
    return q, qi, w


def _run_multi(desc, cache, layer, T, q, qi, w, span_k, span_v, sel=None):
    """GPU: index_topk_multi, csa_decode_multi over its selection (or over the
    given selection), hca_decode_multi. Returns host arrays."""
    B, H, D, k = layer.batch, layer.heads, layer.dim, layer.topk
    ws = dsv4.workspace_multi(desc, T, H, layer.idx_heads, k)
    topk = torch.full((B, T, k), -7, dtype=torch.int32, device="cuda")
    dsv4.dsv4_index_topk_multi(desc, cache, T, layer.idx_heads, to_dev(qi), to_dev(w), k, topk, None, ws)
    use = topk if sel is None else to_dev(sel)
    out = torch.full((B, T, H, D), float("nan"), device="cuda")
    lse = torch.full((B, T, H), float("nan"), device="cuda")
    hout = torch.full((B, T, H, D), float("nan"), device="cuda")
    hlse = torch.full((B, T, H), float("nan"), device="cuda")
    sk, sv = to_dev(span_k), (to_dev(span_v) if span_v is not None else None)
    dsv4.dsv4_csa_decode_multi(desc, cache, T, H, to_dev(q), layer.sm_scale, use, k, sk, sv, out, lse, ws)
    dsv4.dsv4_hca_decode_multi(desc, cache, T, H, to_dev(q), layer.sm_scale, sk, sv, hout, hlse, ws)
    torch.cuda.synchronize()
    assert dsv4.dsv4_read_status(cache) == 0
    return to_host(topk), to_host(out), to_host(lse), to_host(hout), to_host(hlse)


def _check_multi(layer, T, n, planes_of, span_k, span_v, desc, cache, q, qi, w):
    """Selections against the oracle's causal top-k; attention over the
    oracle's selection (uploaded) and, where the selections agree, over the
    chained selection; HCA over the entries complete at each position."""
    o_sel = np.zeros((layer.batch, T, layer.topk), np.int32)
    o_scores = []
    for b in range(layer.batch):
        p = planes_of(b)
        sc = O.index_scores_causal(p["idx_codes"], p["idx_scales"], qi[b], w[b], n, layer.ratio)
        o_scores.append(sc)
        for t in range(T):
            o_sel[b, t] = O.topk_blocks(sc[t], layer.topk)
    g_topk, c_out, c_lse, h_out, h_lse = _run_multi(desc, cache, layer, T, q, qi, w, span_k, span_v)
    _, g_out, g_lse, _, _ = _run_multi(desc, cache, layer, T, q, qi, w, span_k, span_v, sel=o_sel)
    for b in range(layer.batch):
        p = planes_of(b)
        args = (n, layer.ratio, layer.window, p["k_nope"], p["k_scale"], p["k_rope"], span_k[b])
        if layer.separate_v:
            args += (p["v_nope"], p["v_scale"], p["v_rope"], span_v[b])
        oo, ol = O.multi_attend(q[b], np.float32(layer.sm_scale), o_sel[b], *args)
        ho, hl = O.multi_attend(q[b], np.float32(layer.sm_scale), None, *args)
        for t in range(T):
            check_topk(g_topk[b, t], o_scores[b][t], o_sel[b, t], layer.topk)
            assert row_rel_err(g_out[b, t], oo[t]).max() <= TOL, (b, t)
            assert np.abs(g_lse[b, t] - ol[t]).max() <= 1e-3
            if np.array_equal(g_topk[b, t], o_sel[b, t]):
                assert row_rel_err(c_out[b, t], oo[t]).max() <= TOL
            assert row_rel_err(h_out[b, t], ho[t]).max() <= TOL, (b, t)
            assert np.abs(h_lse[b, t] - hl[t]).max() <= 1e-3


@pytest.mark.parametrize("n,T", [(1500, 8), (37, 16), (700, 1)])
def test_multi_token_stream_cache(n, T):
    """A cache built by appending (128 dims, separate V, 4 indexer heads,
    top-64): some queries see fewer blocks than k, the first ones (n = 37)
    fewer tokens than the window."""
    layer = W.scaled(W.CSA_4K, batch=2, n_tokens=n)
    desc, cache = gpu_stream_cache(layer, "multi", T, n, (4096,))
    toks = synth.token_stream("multi", T, layer, layer.batch, 0, n)
    span_k = np.stack([_span(toks["k"][b], n, T, layer.window) for b in range(layer.batch)])
    span_v = np.stack([_span(toks["v"][b], n, T, layer.window) for b in range(layer.batch)])
    q, qi, w = _queries(("multi", n, T), layer, T)
    ocs = [oracle_stream_cache(layer, "multi", T, n, b) for b in range(layer.batch)]
    _check_multi(layer, T, n, lambda b: ocs[b], span_k, span_v, desc, cache, q, qi, w)


def test_multi_token_decode_step_shape():
    """The decode step's layer shape (448 FP8 + 64 BF16 dims, K = V, 64
    heads, 64 indexer heads of 128 dims, top-512, window 128) with 6 queries
    per sequence over directly drawn entries."""
    T = 6
    layer = W.scaled(W.STACK_CSA, batch=2, n_tokens=4 * 2500 + 2)
    planes = oracle_direct_planes(layer, "multistack", 0, range(layer.batch))
    desc, cache = gpu_cache_from_planes(layer, planes)
    n = layer.n_tokens
    span_k = synth.bf16_bits(synth.normal(("multistack", "span"), (layer.batch, T + layer.window - 1, layer.dim)))
    q, qi, w = _queries(("multistack", T), layer, T)
    _check_multi(layer, T, n, lambda b: planes[b], span_k, None, desc, cache, q, qi, w)


def test_multi_token_with_one_query_is_the_single_token_call():
    """T = 1 with a span of the last W tokens gives exactly what the
    single-token calls give on the same cache (the same kernels and plan; the
    window rows read from the span instead of the ring)."""
    layer = W.scaled(W.CSA_4K, batch=2, n_tokens=901)
    n = layer.n_tokens
    desc, cache = gpu_stream_cache(layer, "multi1", 0, n, (4096,))
    toks = synth.token_stream("multi1", 0, layer, layer.batch, 0, n)
    span_k = np.stack([_span(toks["k"][b], n, 1, layer.window) for b in range(layer.batch)])
    span_v = np.stack([_span(toks["v"][b], n, 1, layer.window) for b in range(layer.batch)])
    q, qi, w = _queries(("multi1",), layer, 1)
    m_topk, m_out, m_lse, m_hout, m_hlse = _run_multi(desc, cache, layer, 1, q, qi, w, span_k, span_v)
    B, H, D, k = layer.batch, layer.heads, layer.dim, layer.topk
    ws = dsv4.workspace(desc, H, layer.idx_heads, k)
    topk = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    dsv4.dsv4_index_topk(desc, cache, layer.idx_heads, to_dev(qi[:, 0]), to_dev(w[:, 0]), k, topk, None, ws)
    out = torch.zeros((B, H, D), device="cuda")
    lse = torch.zeros((B, H), device="cuda")
    hout = torch.zeros((B, H, D), device="cuda")
    hlse = torch.zeros((B, H), device="cuda")
    dsv4.dsv4_csa_decode(desc, cache, H, to_dev(q[:, 0]), layer.sm_scale, topk, k, out, lse, ws)
    dsv4.dsv4_hca_decode(desc, cache, H, to_dev(q[:, 0]), layer.sm_scale, hout, hlse, ws)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(topk), m_topk[:, 0])
    assert np.array_equal(to_host(out), m_out[:, 0]) and np.array_equal(to_host(lse), m_lse[:, 0])
    assert np.array_equal(to_host(hout), m_hout[:, 0]) and np.array_equal(to_host(hlse), m_hlse[:, 0])
