"""GPU parity of the projection of the compressor's streams from hidden states
with RoPE (dsv4_project_streams) against the float64 oracle on the same seeded
inputs: every output value within one bf16 step of the oracle's, widened by a
bound on the fp32 accumulation computed from the data, and most values
bit-identical; ragged row counts, a single-token step and positions near 2^20."""
import numpy as np
import pytest
import torch

import oracle as O
from compressed_sparse_kv_05_b300 import dsv4, synth
from compressed_sparse_kv_05_b300 import workloads as W

from .gpu_util import to_dev, to_host

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

BASE = 10000.0


def _bf16_step(v):
    """One bf16 step at each |v| (2^-7 of its binade's lower end)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def _project(layer, T, d_model, n0, tag):
    B, D, Di = layer.batch, layer.dim, layer.idx_dim if layer.kind == "csa" else 0
    h = synth.bf16_bits(synth.normal(tag + ("h",), (B, T, d_model)))
    w = synth.bf16_bits(synth.normal(tag + ("w",), (2 * D + 2 * Di, d_model)) / np.sqrt(d_model))
    desc = dsv4.layer_desc(layer, 64)
    cache = dsv4.Cache(desc)
    cache.n_tokens.copy_(torch.tensor(n0, dtype=torch.int64))
    x = torch.full((B, T, D), -1, dtype=torch.int16, device="cuda")
    z = torch.full((B, T, D), -1, dtype=torch.int16, device="cuda")
    u = torch.full((B, T, max(Di, 1)), -1, dtype=torch.int16, device="cuda")
    zu = torch.full((B, T, max(Di, 1)), -1, dtype=torch.int16, device="cuda")
    dsv4.dsv4_project_streams(desc, cache, T, d_model, to_dev(h), to_dev(w), BASE, x, z,
                              u if Di else None, zu if Di else None)
    torch.cuda.synchronize()
    assert dsv4.dsv4_read_status(cache) == 0
    g = [to_host(t, np.uint16) for t in (x, z, u, zu)]
    return h, w, g, Di


def _check(layer, T, d_model, n0, tag):
    h, w, g, Di = _project(layer, T, d_model, n0, tag)
    D = layer.dim
    wf = O.bf16_decode(w)
    exact = total = 0
    for b in range(layer.batch):
        pos = n0[b] + np.arange(T)
        o = O.project_streams(h[b], w, layer.d_nope, layer.d_rope, Di, pos, BASE)
        S = np.abs(O.bf16_decode(h[b])) @ np.abs(wf).T        # sum |h| |w| per (row, column)
        acc = S * d_model * 2.0 ** -23                          # fp32 accumulation, generously
        # a rotated value mixes its pair: take the pair's larger bound, plus the rotation's rounding
        cols = [(0, D), (D, 2 * D), (2 * D, 2 * D + Di), (2 * D + Di, 2 * D + 2 * Di)]
        for s, (c0, c1) in enumerate(cols[:4 if Di else 2]):
            ov = O.bf16_decode(o[s])
            gv = O.bf16_decode(g[s][b][:, :c1 - c0])
            bound = acc[:, c0:c1].copy()
            pair = np.maximum(bound[:, 0::2], bound[:, 1::2])
            bound[:, 0::2] = pair
            bound[:, 1::2] = pair
            bound += 2.0 ** -21 * np.abs(ov)
            err = np.abs(gv - ov)
            assert np.all(err <= _bf16_step(ov) + bound), (b, s, float((err - _bf16_step(ov) - bound).max()))
            exact += int(np.sum(g[s][b][:, :c1 - c0] == o[s]))
            total += ov.size
    print(f"bit-identical to the oracle: {exact} of {total}")
    assert exact >= 0.97 * total


@pytest.mark.parametrize("T,n0", [(130, (0, 1_000_000)), (1, (5, 1 << 20)), (300, (77, 4096))])
def test_project_streams_decode_step_shape(T, n0):
    """The decode step's CSA layer dims (448 + 64, 128-dim indexer keys), a
    512-wide hidden state, B = 2: 130 tokens (two 128-row tiles, the second
    ragged), one token, and 300 tokens."""
    layer = W.scaled(W.STACK_CSA, batch=2)
    _check(layer, T, 512, n0, ("proj", T))


def test_project_streams_small_layer_without_indexer():
    """A 64 + 64 HCA layer (no indexer streams), 192-wide hidden state, 4 sequences."""
    layer = W.Layer("hca", 4, 0, 8, 64, 64, False, 128, 128)
    _check(layer, 70, 192, (0, 1, 1000, 123456), ("proj_small",))


def test_project_streams_zero_tokens_and_unsupported_shapes():
    layer = W.scaled(W.STACK_CSA, batch=1)
    desc = dsv4.layer_desc(layer, 64)
    cache = dsv4.Cache(desc)
    x = torch.zeros((1, 1, layer.dim), dtype=torch.int16, device="cuda")
    dsv4.dsv4_project_streams(desc, cache, 0, 512, x, x, BASE, x, x, x, x)
    for d_model in (100, 0):
        with pytest.raises(RuntimeError):
            dsv4.dsv4_project_streams(desc, cache, 1, d_model, x, x, BASE, x, x, x, x)


def test_project_streams_chunk_shape_and_full_width_tiles():
    """The tile width follows the call's shape (it fills the SMs' waves): a
    4096-token call of the decode step's layer (1280 columns) takes 160-column
    tiles on 148 SMs; 18944 tokens of a 256-column layer take 256-column tiles."""
    _check(W.scaled(W.STACK_CSA, batch=1), 4096, 256, (100000,), ("proj_chunk",))
    _check(W.Layer("hca", 1, 0, 8, 64, 64, False, 128, 128), 18944, 128, (3,), ("proj_wide",))


def test_projection_feeds_single_token_appends_in_stream():
    """The streams the projection writes are what the compressor reads: one
    token at a time, projection then append, back to back on one stream with
    no synchronisation (each kernel may start while the one before it
    finishes) gives the same cache bytes as the same calls each followed by a
    device synchronisation."""
    layer = W.scaled(W.STACK_CSA, batch=2)
    B, D, Di, d_model, steps = layer.batch, layer.dim, layer.idx_dim, 512, 48
    h = to_dev(synth.bf16_bits(synth.normal(("chain", "h"), (steps, B, 1, d_model))))
    w = to_dev(synth.bf16_bits(synth.normal(("chain", "w"), (2 * D + 2 * Di, d_model)) / np.sqrt(d_model)))
    b = to_dev(synth.position_bias("chain", 0, layer, "b"))
    bu = to_dev(synth.position_bias("chain", 0, layer, "bu"))
    desc = dsv4.layer_desc(layer, 64)
    caches = []
    for sync in (False, True):
        cache = dsv4.Cache(desc)
        x, z = (torch.zeros((B, 1, D), dtype=torch.int16, device="cuda") for _ in range(2))
        u, zu = (torch.zeros((B, 1, Di), dtype=torch.int16, device="cuda") for _ in range(2))
        for s in range(steps):
            dsv4.dsv4_project_streams(desc, cache, 1, d_model, h[s], w, BASE, x, z, u, zu)
            if sync:
                torch.cuda.synchronize()
            dsv4.dsv4_compress_append(desc, cache, 1, x, None, z, b, u, zu, bu)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        assert dsv4.dsv4_read_status(cache) == 0
        caches.append(cache)
    assert int(caches[0].n_tokens[0]) == steps
    for name, t in vars(caches[1]).items():
        if isinstance(t, torch.Tensor):
            assert torch.equal(getattr(caches[0], name), t), name
