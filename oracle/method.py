"""Float64 CPU statement of CSA / HCA decode over a low-bit compressed KV cache.

TEST INFRASTRUCTURE ONLY (see ``oracle/formats.py``): importable from tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` only.

What the pages fix, and where (titles and sections of the source pages):
  [HYB] vibecoco.ai, "DeepSeek V4 agent architecture", section
        "混合注意力：两种压缩，交替使用" (hybrid attention, two compressions used
        alternately). CSA pools KV along the sequence 4:1 with softmax-gated
        pooling plus a learned position bias; a lightning indexer (multi-head
        dot products scored through ReLU, run in FP4) picks the top-k compressed
        blocks; recent tokens keep full precision in a sliding-window branch.
        HCA pools 128:1 and every query attends densely to all compressed
        entries. Entries are FP8 except the RoPE dims, which stay BF16.
  [CSA] pnsm.cn, "DeepSeek V4 架构深度解析：百万Token上下文背后的技术革命与Agent生态重构",
        section 2.1 "CSA：压缩稀疏注意力": two KV paths, a sliding window kept
        as a ring of window_size entries overwritten cyclically, and a
        compressor whose outputs are filtered to the top-k by an index.
  [HCA] same page, section 2.2 "HCA：重度压缩注意力": 128:1 compression,
        alternating with CSA across layers.
  [ROPE] devpress.csdn.net, "DeepSeek-V4：百万Token上下文，这次智能体真的能用了",
        section "二、DeepSeek-V4的核心架构创新", part "位置编码的长度泛化优化":
        positions enter through RoPE, extended to long contexts by training
        (no inference-time change to the rotation is described).

Readings taken where the pages leave a step open (the plainest one the rest
supports):
  * pooling is along the sequence over non-overlapping blocks [j*m, (j+1)*m);
    the weights are a per-channel softmax over the m tokens of (gate logit +
    position bias); an incomplete trailing block is not emitted;
  * one gate stream gates both K and V of a token; the indexer keys are a
    separate per-token stream pooled the same way with their own gates/bias;
  * an FP8 entry stores codes of y/s with s = amax(|y_nope|)/448 (fp32), the
    RoPE dims as bf16; FP4 rows use blocks of 16 with an e4m3 scale
    e4m3(amax/6); the quantisation decisions are made in fp32 on the pooled
    value rounded to fp32;
  * indexer score I_s = sum_h w_h * max(0, q_h . k_s) on exactly decoded FP4
    query and key; top-k ties go to the lower block index and the selection is
    returned in ascending index order, padded with -1;
  * attention is one softmax over (selected compressed entries) U (window
    tokens); the window holds the last min(W, n) raw bf16 tokens and is not
    masked against the compressed blocks it overlaps; the query is used
    exactly as given (bf16); V = K for a shared entry;
  * the streams the compressor pools (token keys x, gate logits z, indexer keys
    u and their gates zu) are linear projections of the hidden state ([HYB]:
    the pooling is learned); RoPE is the standard rotation: pairs (2i, 2i + 1)
    of the rotated dims turn by pos * base^(-2i/d), applied to the trailing
    d_rope dims of x and the trailing min(d_rope, Di) dims of u at each
    token's absolute position, before pooling and before the window ring; each
    projected stream is rounded once to bf16 (the compressor's input format).
"""
import numpy as np

from .formats import (bf16_decode, bf16_encode, e2m1_decode, e2m1_encode,
                      e4m3_decode, e4m3_encode)

# ----------------------------------------------------------------------------- pooling


def pool_blocks(x_bits, z_bits, bias, ratio):
    """Softmax-gated pooling along the sequence [HYB].

    x_bits, z_bits : uint16 bf16 [T][C] token values and gate logits
    bias           : float32 [ratio][C] learned position bias, added to the logits
    returns float32 [T // ratio][C]: for block j and channel c,
        y[j, c] = sum_i softmax_i(z[j*m+i, c] + b[i, c]) * x[j*m+i, c]
    computed in float64 and rounded once to float32.
    """
    x = bf16_decode(x_bits)
    z = bf16_decode(z_bits)
    T, C = x.shape
    nb = T // ratio
    if nb == 0:
        return np.zeros((0, C), np.float32)
    x = x[: nb * ratio].reshape(nb, ratio, C)
    logits = z[: nb * ratio].reshape(nb, ratio, C) + np.asarray(bias, np.float32).astype(np.float64)[None]
    logits = logits - logits.max(axis=1, keepdims=True)
    w = np.exp(logits)
    w = w / w.sum(axis=1, keepdims=True)
    return (w * x).sum(axis=1).astype(np.float32)


# ----------------------------------------------------------------------------- quantisation


def quantize_kv_rows(y, d_nope):
    """FP8 entry with BF16 RoPE dims [HYB].

    y : float32 [R][d_nope + d_rope] pooled rows.
    returns (nope uint8 [R][d_nope] e4m3 codes, scale float32 [R], rope uint16 [R][d_rope] bf16)
    with s = amax/448 and code = e4m3(y/s), both divisions in IEEE fp32; s = 0
    (an all-zero row) gives all-zero codes.
    """
    y = np.asarray(y, np.float32)
    yn = y[:, :d_nope]
    amax = np.abs(yn).max(axis=1, initial=np.float32(0))
    s = (amax / np.float32(448.0)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = (yn / safe[:, None]).astype(np.float32)
    codes = e4m3_encode(q)
    codes[s == 0] = 0
    return codes, s, bf16_encode(y[:, d_nope:])


def quantize_fp4_rows(y):
    """FP4 rows with one e4m3 scale per 16 contiguous values [HYB].

    y : float32 [R][C], C a multiple of 16.
    returns (codes uint8 [R][C/2] with element 2i in the low nibble, scales uint8 [R][C/16])
    with scale = e4m3(amax/6) and code = e2m1(y/scale), fp32 divisions; a zero
    scale gives zero codes.
    """
    y = np.asarray(y, np.float32)
    R, C = y.shape
    blocks = y.reshape(R, C // 16, 16)
    amax = np.abs(blocks).max(axis=2, initial=np.float32(0))
    s_code = e4m3_encode((amax / np.float32(6.0)).astype(np.float32))
    s = e4m3_decode(s_code).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = (blocks / safe[:, :, None]).astype(np.float32)
    c = e2m1_encode(q)
    c[s == 0] = 0
    c = c.reshape(R, C)
    packed = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    return packed, s_code


def dequant_kv_rows(nope, scale, rope):
    """Exact float64 value of FP8+BF16 entries: [code * s || rope]."""
    return np.concatenate([e4m3_decode(nope) * np.asarray(scale, np.float32).astype(np.float64)[:, None],
                           bf16_decode(rope)], axis=1)


def dequant_fp4_rows(codes, scales):
    """Exact float64 value of FP4 rows: e2m1(code) * e4m3(scale) per block of 16."""
    codes = np.asarray(codes, np.uint8)
    R, half = codes.shape
    C = half * 2
    vals = np.empty((R, C), np.float64)
    vals[:, 0::2] = e2m1_decode(codes & 0xF)
    vals[:, 1::2] = e2m1_decode(codes >> 4)
    s = e4m3_decode(scales).reshape(R, C // 16)
    return (vals.reshape(R, C // 16, 16) * s[:, :, None]).reshape(R, C)


# ----------------------------------------------------------------------------- cache


def build_cache(k_bits, z_bits, bias, ratio, d_nope, window, v_bits=None,
                u_bits=None, zu_bits=None, bias_u=None):
    """Cache of ONE sequence after its first n tokens have been appended.

    k_bits, z_bits [n][D] (and v_bits [n][D] when K and V are separate) are the
    raw bf16 tokens and gate logits; u_bits, zu_bits [n][Di] the indexer-key
    stream. Returns a dict with, for the n // ratio complete blocks, the pooled
    fp32 rows and their quantised planes; the window ring (token t in slot
    t % window, the last min(window, n) tokens); the tokens of the open block
    (slot t % ratio) [CSA].
    """
    n = k_bits.shape[0]
    out = {"n_tokens": n}
    yk = pool_blocks(k_bits, z_bits, bias, ratio)
    out["pooled_k"] = yk
    out["k_nope"], out["k_scale"], out["k_rope"] = quantize_kv_rows(yk, d_nope)
    if v_bits is not None:
        yv = pool_blocks(v_bits, z_bits, bias, ratio)
        out["pooled_v"] = yv
        out["v_nope"], out["v_scale"], out["v_rope"] = quantize_kv_rows(yv, d_nope)
    if u_bits is not None:
        yu = pool_blocks(u_bits, zu_bits, bias_u, ratio)
        out["pooled_u"] = yu
        out["idx_codes"], out["idx_scales"] = quantize_fp4_rows(yu)
    first = max(0, n - window)
    ring_slots = {}
    for t in range(first, n):
        ring_slots[t % window] = t
    out["ring_slots"] = ring_slots          # slot -> token position
    out["win_k"] = {s: k_bits[t] for s, t in ring_slots.items()}
    if v_bits is not None:
        out["win_v"] = {s: v_bits[t] for s, t in ring_slots.items()}
    open_first = (n // ratio) * ratio
    out["pending"] = {t % ratio: t for t in range(open_first, n)}
    return out


def window_tokens(n, window):
    """Positions held by the window after n tokens: the last min(window, n)."""
    return np.arange(max(0, n - window), n)


# ----------------------------------------------------------------------------- indexer


def index_scores(idx_codes, idx_scales, q_idx_bits, w):
    """Lightning-indexer scores of one sequence [HYB].

    idx_codes/idx_scales : FP4 keys [n_c][Di/2], [n_c][Di/16]
    q_idx_bits           : bf16 [Hi][Di] indexer query, quantised to FP4 with
                           the same rule as the keys (the indexer runs in FP4)
    w                    : float32 [Hi] head weights
    returns float64 [n_c]: I_s = sum_h w_h * max(0, q_h . k_s) on decoded values.
    """
    qc, qs = quantize_fp4_rows(bf16_decode(q_idx_bits).astype(np.float32))
    Q = dequant_fp4_rows(qc, qs)
    K = dequant_fp4_rows(idx_codes, idx_scales)
    dots = K @ Q.T
    return (np.maximum(dots, 0.0) * np.asarray(w, np.float32).astype(np.float64)[None, :]).sum(axis=1)


def topk_blocks(scores, k):
    """Indices of the k largest scores; ties -> lower index; ascending order;
    -1 padding when fewer than k blocks exist [HYB], [CSA]."""
    scores = np.asarray(scores, np.float64)
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores))
    sel = np.sort(order[: min(k, n)]).astype(np.int32)
    return np.concatenate([sel, np.full(k - sel.shape[0], -1, np.int32)])


def topk_boundary_gap(scores, k):
    """Relative gap (I_(k) - I_(k+1)) / |I_(k)| between the k-th and (k+1)-th
    largest scores. +inf when there is no (k+1)-th score; 0 for an exact tie."""
    s = np.sort(np.asarray(scores, np.float64))[::-1]
    if s.shape[0] <= k:
        return np.inf
    a, b = s[k - 1], s[k]
    if a == b:
        return 0.0
    return (a - b) / abs(a)


# ----------------------------------------------------------------------------- attention


def attend(q_bits, K, V, sm_scale):
    """One softmax over all rows of K/V for every query head.

    q_bits : bf16 [H][D]; K float64 [N][D]; V float64 [N][Dv]; sm_scale fp32.
    returns (out float64 [H][Dv], lse float64 [H], natural log). N = 0 gives
    out = 0 and lse = -inf.
    """
    q = bf16_decode(q_bits)
    H = q.shape[0]
    if K.shape[0] == 0:
        return np.zeros((H, V.shape[1])), np.full(H, -np.inf)
    s = float(np.float32(sm_scale)) * (q @ K.T)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    return (p @ V) / l, (m + np.log(l))[:, 0]


def lse_merge(outs, lses):
    """Combine attention partials over disjoint row sets into the attention over
    their union: o = sum_p exp(lse_p - lse) o_p with lse = log sum_p exp(lse_p)."""
    lses = np.asarray(lses, np.float64)
    outs = np.asarray(outs, np.float64)
    m = lses.max(axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    wts = np.exp(lses - m_safe[None])
    tot = wts.sum(axis=0)
    lse = np.where(tot > 0, m_safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    out = (wts[..., None] * outs).sum(axis=0) / np.where(tot > 0, tot, 1.0)[..., None]
    return out, lse


def _window_rows(win_ring, n, window, dim):
    """float64 rows of the window, oldest first, read from a bf16 ring [W][dim]."""
    pos = window_tokens(n, window)
    if pos.shape[0] == 0:
        return np.zeros((0, dim))
    return bf16_decode(win_ring[pos % window])


def csa_attend(q_bits, sm_scale, topk, n_tokens, ratio, window,
               k_nope, k_scale, k_rope, win_k,
               v_nope=None, v_scale=None, v_rope=None, win_v=None):
    """CSA decode for one sequence [HYB], [CSA]: attention of q over the top-k
    compressed entries together with the raw window, under one softmax.
    topk entries equal to -1 are padding. Cache planes are this sequence's."""
    n_c = n_tokens // ratio
    sel = np.asarray([i for i in np.asarray(topk).tolist() if i >= 0], np.int64)
    if np.any(sel >= n_c):
        raise ValueError("top-k index beyond the compressed entries")
    K = dequant_kv_rows(k_nope[sel], k_scale[sel], k_rope[sel])
    Kall = np.concatenate([K, _window_rows(win_k, n_tokens, window, K.shape[1])], axis=0)
    if v_nope is None:
        Vall = Kall
    else:
        V = dequant_kv_rows(v_nope[sel], v_scale[sel], v_rope[sel])
        Vall = np.concatenate([V, _window_rows(win_v, n_tokens, window, V.shape[1])], axis=0)
    return attend(q_bits, Kall, Vall, sm_scale)


def hca_attend(q_bits, sm_scale, n_tokens, ratio, window,
               k_nope, k_scale, k_rope, win_k,
               v_nope=None, v_scale=None, v_rope=None, win_v=None):
    """HCA decode for one sequence [HYB], [HCA]: dense attention over every
    compressed entry together with the raw window, under one softmax."""
    n_c = n_tokens // ratio
    all_idx = np.arange(n_c, dtype=np.int32)
    return csa_attend(q_bits, sm_scale, all_idx, n_tokens, ratio, window,
                      k_nope, k_scale, k_rope, win_k, v_nope, v_scale, v_rope, win_v)


# ----------------------------------------------------------------------------- several queries per step


def query_positions(n_tokens, T):
    """Positions of the T queries of a multi-token step taken after their T
    tokens were appended to a sequence of n_tokens tokens: n - T + t [CSA]."""
    return np.arange(n_tokens - T, n_tokens)


def index_scores_causal(idx_codes, idx_scales, q_idx_bits, w, n_tokens, ratio):
    """Lightning-indexer scores of T queries [HYB], [CSA], each over the
    compressed blocks complete at its own position (a causal selection): query
    t at position p scores blocks j < (p + 1) // ratio, with its own indexer
    query q_idx_bits[t] (bf16 [Hi][Di]) and head weights w[t].
    Returns a list of T float64 arrays (scores of blocks 0 .. n_c(t) - 1)."""
    T = q_idx_bits.shape[0]
    out = []
    for t, p in enumerate(query_positions(n_tokens, T)):
        n_c = (p + 1) // ratio
        out.append(index_scores(idx_codes[:n_c], idx_scales[:n_c], q_idx_bits[t], w[t]))
    return out


def multi_attend(q_bits, sm_scale, sel, n_tokens, ratio, window, k_nope, k_scale, k_rope, span_k,
                 v_nope=None, v_scale=None, v_rope=None, span_v=None):
    """Attention of T queries of one sequence [HYB], [CSA], [HCA]: query t at
    position p = n - T + t attends, under one softmax, to the compressed
    entries sel[t] (indices < (p + 1) // ratio; -1 is padding), or to every
    entry complete by p when sel is None, together with the raw tokens of the
    positions max(0, p - W + 1) .. p. span_k (span_v) holds the raw rows of the
    positions n - T - W + 1 .. n - 1, row r for position n - T - W + 1 + r.
    Returns (out [T][H][Dv], lse [T][H])."""
    T = q_bits.shape[0]
    first = n_tokens - T - window + 1          # position of span row 0
    outs, lses = [], []
    for t, p in enumerate(query_positions(n_tokens, T)):
        n_c = (p + 1) // ratio
        idx = np.arange(n_c) if sel is None else np.asarray([i for i in np.asarray(sel[t]).tolist() if i >= 0])
        if np.any(idx >= n_c):
            raise ValueError("a selected entry is not complete at the query's position")
        idx = idx.astype(np.int64)
        pos = np.arange(max(0, p - window + 1), p + 1)
        K = np.concatenate([dequant_kv_rows(k_nope[idx], k_scale[idx], k_rope[idx]),
                            bf16_decode(span_k[pos - first]) if pos.size else
                            np.zeros((0, k_nope.shape[1] + k_rope.shape[1]))], axis=0)
        if v_nope is None:
            V = K
        else:
            V = np.concatenate([dequant_kv_rows(v_nope[idx], v_scale[idx], v_rope[idx]),
                                bf16_decode(span_v[pos - first]) if pos.size else
                                np.zeros((0, v_nope.shape[1] + v_rope.shape[1]))], axis=0)
        o, l = attend(q_bits[t], K, V, sm_scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def rope_rotate(x, pos, base):
    """RoPE [ROPE] of the rows of x (float64, d even columns) at positions pos
    (one per row): pair (2i, 2i + 1) turns by the angle pos * base^(-2i/d),
    (a, b) -> (a cos - b sin, a sin + b cos)."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    theta = float(base) ** (-2.0 * np.arange(d // 2) / d)
    ang = np.asarray(pos, np.float64).reshape(-1, 1) * theta[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def project_streams(h_bits, w_bits, d_nope, d_rope, idx_dim, pos, base):
    """The compressor's input streams of T tokens from their hidden states
    ([HYB] learned pooling, [ROPE]): y = h . W^T over the bf16 operands in
    float64, W's rows being x (D = d_nope + d_rope), z (D), u (idx_dim), zu
    (idx_dim) in that order; RoPE at the tokens' positions on the trailing
    d_rope dims of x and the trailing min(d_rope, idx_dim) dims of u; each
    stream rounded once to bf16. Returns the bf16 bit patterns (x, z, u, zu),
    u and zu with idx_dim columns (zero columns when idx_dim is 0)."""
    h = bf16_decode(h_bits)
    w = bf16_decode(w_bits)
    D = d_nope + d_rope
    if w.shape[0] != 2 * D + 2 * idx_dim or w.shape[1] != h.shape[1]:
        raise ValueError("weight rows must be 2 (d_nope + d_rope) + 2 idx_dim, columns the hidden size")
    y = h @ w.T
    x = y[:, :D].copy()
    z = y[:, D:2 * D]
    u = y[:, 2 * D:2 * D + idx_dim].copy()
    zu = y[:, 2 * D + idx_dim:]
    if d_rope:
        x[:, d_nope:] = rope_rotate(x[:, d_nope:], pos, base)
    ur = min(d_rope, idx_dim)
    if ur:
        u[:, idx_dim - ur:] = rope_rotate(u[:, idx_dim - ur:], pos, base)
    return tuple(bf16_encode(a) for a in (x, z, u, zu))
