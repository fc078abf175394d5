"""Byte accounting of the compressed cache and of one decode step.

Bytes counted per decode step are only those the method has to move (the
algorithmic bytes): all indexer keys (CSA), the selected top-k entries (CSA) or
every compressed entry (HCA), the window tokens, the queries, the indexer query
and weights, and the output. Intermediates (scores, split partials, top-k
indices) are not counted.
"""


def entry_bytes(layer):
    """Bytes of one compressed KV entry: FP8 codes + fp32 scale + BF16 RoPE dims
    (twice when K and V are stored separately)."""
    one = layer.d_nope + 4 + 2 * layer.d_rope
    return one * (2 if layer.separate_v else 1)


def idx_key_bytes(layer):
    """Bytes of one FP4 indexer key: Di/2 code bytes + Di/16 e4m3 scales."""
    return layer.idx_dim // 2 + layer.idx_dim // 16 if layer.idx_dim else 0


def kv_bytes_per_token(layer):
    """Cache bytes per context token for this layer kind (window excluded)."""
    return (entry_bytes(layer) + (idx_key_bytes(layer) if layer.kind == "csa" else 0)) / layer.ratio


def gqa_bf16_bytes_per_token(kv_heads=8, head_dim=128):
    """Per-token K+V bytes of a bf16 grouped-query-attention layer."""
    return 2 * kv_heads * head_dim * 2


def decode_step_bytes(layer, n_tokens=None):
    """Algorithmic bytes one decode step of one layer moves, all sequences."""
    n = layer.n_tokens if n_tokens is None else n_tokens
    n_c = n // layer.ratio
    per_kv = 2 if layer.separate_v else 1
    win = min(layer.window, n) * layer.dim * 2 * per_kv
    q = layer.heads * layer.dim * 2
    out = layer.heads * layer.dim * 4
    if layer.kind == "csa":
        sel = min(layer.topk, n_c) * entry_bytes(layer)
        idx = n_c * idx_key_bytes(layer) + layer.idx_heads * layer.idx_dim * 2 + layer.idx_heads * 4
        body = idx + sel
    else:
        body = n_c * entry_bytes(layer)
    return layer.batch * (body + win + q + out)


def call_bytes(layer, call, n_tokens=None):
    """Algorithmic bytes of one library call of one decode step (all sequences).

    append      : the new token's k, z (v, u, zu) read + its window-ring and
                  pending writes, plus the entry written when it completes a
                  block (amortised: one in `ratio` steps)
    index_topk  : all indexer keys + indexer query and weights + top-k indices written
    csa_decode  : selected entries + window + query + output
    hca_decode  : every entry + window + query + output
    """
    n = layer.n_tokens if n_tokens is None else n_tokens
    n_c = n // layer.ratio
    B = layer.batch
    per_kv = 2 if layer.separate_v else 1
    D = layer.dim
    win = min(layer.window, n) * D * 2 * per_kv
    q = layer.heads * D * 2
    out = layer.heads * D * 4
    if call == "append":
        tok = D * 2 * (1 + per_kv) + (2 * layer.idx_dim * 2 if layer.kind == "csa" else 0)
        writes = D * 2 * per_kv * 2 + (2 * layer.idx_dim * 2 if layer.kind == "csa" else 0)
        entry = (entry_bytes(layer) + (idx_key_bytes(layer) if layer.kind == "csa" else 0)) / layer.ratio
        return B * (tok + writes + entry)
    if call == "index_topk":
        return B * (n_c * idx_key_bytes(layer) + layer.idx_heads * layer.idx_dim * 2 + layer.idx_heads * 4
                    + layer.topk * 4)
    if call == "csa_decode":
        return B * (min(layer.topk, n_c) * entry_bytes(layer) + win + q + out)
    if call == "hca_decode":
        return B * (n_c * entry_bytes(layer) + win + q + out)
    raise ValueError(call)
