"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module draws random numbers and casts them to the input dtypes; it holds
none of the method's arithmetic (no pooling, quantisation, scoring, selection or
attention). Every tensor is identified by (seed, workload tag, layer, tensor
name) and drawn from numpy's PCG64 seeded by a SeedSequence over those parts, so
any process that asks for the same tensor gets the same bytes.

bf16 inputs are float32 draws cast to bfloat16 by torch (round to nearest even).
"""
import zlib

import numpy as np
import torch

BASE_SEED = 0


def _parts(parts):
    out = []
    for p in parts:
        out.append(zlib.crc32(p.encode()) if isinstance(p, str) else int(p))
    return out


def rng(*parts):
    """numpy Generator for one named tensor."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(_parts((BASE_SEED,) + parts))))


def normal(parts, shape, std=1.0):
    a = rng(*parts).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def uniform(parts, shape, lo=0.0, hi=1.0):
    return rng(*parts).uniform(lo, hi, size=shape).astype(np.float32)


def bf16_bits(a):
    """float32 array -> uint16 array of bfloat16 bit patterns (torch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------- token streams


def token_stream(tag, layer_id, layer, batch, t0, t1):
    """Tokens [t0, t1) of every sequence, for appending to a layer's cache.

    Returns a dict of bf16 bit arrays k, z (and v when K and V are separate;
    u, zu when the layer has an indexer), each [batch][t1 - t0][dims]. Each
    sequence's stream is drawn once per (tag, layer, sequence, tensor) in
    blocks of 4096 tokens, so any [t0, t1) slice of it is the same bytes
    whatever the chunking.
    """
    out = {}
    names = [("k", layer.dim), ("z", layer.dim)]
    if layer.separate_v:
        names.append(("v", layer.dim))
    if layer.idx_dim:
        names += [("u", layer.idx_dim), ("zu", layer.idx_dim)]
    for name, dim in names:
        arr = np.empty((batch, t1 - t0, dim), np.uint16)
        for b in range(batch):
            arr[b] = _stream_slice((tag, layer_id, b, name), dim, t0, t1)
        out[name] = arr
    return out


_STREAM_BLOCK = 4096


def _stream_slice(parts, dim, t0, t1):
    if t1 <= t0:
        return np.zeros((0, dim), np.uint16)
    first, last = t0 // _STREAM_BLOCK, (t1 - 1) // _STREAM_BLOCK
    full = np.concatenate([bf16_bits(normal(parts + ("blk", blk), (_STREAM_BLOCK, dim)))
                           for blk in range(first, last + 1)], axis=0)
    off = first * _STREAM_BLOCK
    return full[t0 - off: t1 - off]


def position_bias(tag, layer_id, layer, name="b"):
    """Learned position bias stand-in, ~N(0, 0.1), float32 [ratio][dims]."""
    dim = layer.idx_dim if name == "bu" else layer.dim
    return normal((tag, layer_id, name), (layer.ratio, dim), std=0.1)


# ----------------------------------------------------------------------------- decode inputs


def decode_inputs(tag, layer_id, layer, step=0):
    """Per-step decode inputs of one layer: q bf16 [B][H][D]; for CSA also the
    indexer query q_idx bf16 [B][Hi][Di] and head weights w ~U(0,1) float32 [B][Hi]."""
    B = layer.batch
    out = {"q": bf16_bits(normal((tag, layer_id, "q", step), (B, layer.heads, layer.dim)))}
    if layer.kind == "csa":
        out["q_idx"] = bf16_bits(normal((tag, layer_id, "q_idx", step), (B, layer.idx_heads, layer.idx_dim)))
        out["w"] = uniform((tag, layer_id, "w", step), (B, layer.idx_heads))
    return out


# ----------------------------------------------------------------------------- directly drawn caches


def direct_rows(tag, layer_id, layer, b):
    """Pooled rows of one sequence, drawn directly instead of pooled from tokens.

    Returns float32 kv [n_comp][D] ~N(0,1), and for CSA idx [n_comp][Di]
    ~N(0,1) in which a fraction of the blocks (planted_frac, at least one) is
    replaced by a key aligned with the step-0 indexer query: 4 * qbar / rms(qbar)
    with qbar = sum_h w_h q_idx[h], so that the top-k has real winners. Also
    returns the planted block indices.
    """
    n_c = layer.n_comp
    kv = normal((tag, layer_id, b, "kv_rows"), (n_c, layer.dim))
    res = {"kv": kv}
    if layer.separate_v:
        res["v"] = normal((tag, layer_id, b, "v_rows"), (n_c, layer.dim))
    if layer.kind == "csa":
        idx = normal((tag, layer_id, b, "idx_rows"), (n_c, layer.idx_dim))
        planted = np.zeros(0, np.int64)
        if layer.planted_frac > 0 and n_c > 0:
            cnt = max(1, int(np.ceil(layer.planted_frac * n_c)))
            planted = np.sort(rng(tag, layer_id, b, "planted").choice(n_c, size=min(cnt, n_c), replace=False))
            dec = decode_inputs(tag, layer_id, layer, 0)
            qi = torch.from_numpy(dec["q_idx"][b].view(np.int16)).view(torch.bfloat16).float().numpy()
            qbar = (dec["w"][b][:, None] * qi).sum(axis=0)
            rms = np.sqrt(np.mean(qbar.astype(np.float64) ** 2))
            idx[planted] = (4.0 * qbar / rms).astype(np.float32)[None, :]
        res["idx"] = idx
        res["planted"] = planted
    return res


def window_tokens(tag, layer_id, layer, b):
    """The raw bf16 tokens at positions [n - W, n) of a directly drawn cache,
    oldest first: dict with k (and v) [min(W, n)][D]."""
    cnt = min(layer.window, layer.n_tokens)
    out = {"k": bf16_bits(normal((tag, layer_id, b, "win_k"), (cnt, layer.dim)))}
    if layer.separate_v:
        out["v"] = bf16_bits(normal((tag, layer_id, b, "win_v"), (cnt, layer.dim)))
    return out
