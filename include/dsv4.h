/*
 * dsv4.h -- C ABI of libdsv4: single-token decode through CSA / HCA attention
 * layers over a KV cache held in FP8 / BF16 / FP4, on one B300 (sm_103a).
 *
 * The method (titles and sections of the pages that describe it):
 *   [HYB] vibecoco.ai, "DeepSeek V4 agent architecture", section
 *         "混合注意力：两种压缩，交替使用" (hybrid attention): CSA compresses the
 *         KV entries 4:1 along the sequence by softmax-gated pooling with a
 *         learned position bias, scores the compressed blocks with an FP4
 *         lightning indexer (multi-head dot products through ReLU), keeps the
 *         top-k blocks and adds a sliding window of recent raw tokens; HCA
 *         compresses 128:1 and attends densely to every compressed entry.
 *         Entries are FP8 except the RoPE dims, kept in BF16.
 *   [CSA] pnsm.cn, "DeepSeek V4 架构深度解析：百万Token上下文背后的技术革命与
 *         Agent生态重构", section 2.1 "CSA：压缩稀疏注意力": a window ring of
 *         window_size entries overwritten cyclically, and a compressor whose
 *         outputs are filtered to the top-k by an index.
 *   [HCA] same page, section 2.2 "HCA：重度压缩注意力".
 *   [ROPE] devpress.csdn.net, "DeepSeek-V4：百万Token上下文，这次智能体真的能用了",
 *         section "二、DeepSeek-V4的核心架构创新", part "位置编码的长度泛化优化":
 *         positions enter through RoPE.
 *
 * Conventions shared by every call
 *   - Data pointers are DEVICE pointers owned by the caller (the library never
 *     allocates, frees or keeps them). Every plane must start on a 16-byte
 *     boundary.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call
 *     only enqueues work on it and returns; results are ready when the stream
 *     reaches that point. Calls on different caches may run concurrently.
 *   - Kernels are launched as programmatic dependent launches: each may start
 *     while the kernel before it in the stream finishes, and waits for that
 *     kernel before it reads anything it may have written. A few inputs are
 *     read before that wait: the attention query `q` of dsv4_csa_decode(_multi)
 *     and dsv4_hca_decode(_static), the indexer query `q_idx` and weights `w`
 *     of dsv4_index_topk(_multi). They must be complete when the call is
 *     enqueued in stream order, i.e. written by work that is not a kernel of
 *     this library still running in the same stream (a projection GEMM or a
 *     copy enqueued before the call qualifies, unless it triggers
 *     programmatic launch of its dependents before those writes; the `out` of
 *     a call enqueued just before does not). The streams dsv4_project_streams
 *     writes are read by dsv4_compress_append after its wait.
 *   - Return value: DSV4_OK, or a negative DSV4_ERR_* code. A call that
 *     returns an error found on the host launches nothing and changes nothing.
 *     Conditions only the device can see (capacity, bad indices) set bits of
 *     the cache's device status word, read with dsv4_read_status().
 *   - bf16 values travel as uint16_t bit patterns, FP8 as e4m3 (OCP "e4m3fn")
 *     bytes, FP4 as e2m1 nibbles two to a byte (element 2i in the low nibble).
 */
#ifndef DSV4_H
#define DSV4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  DSV4_OK = 0,
  DSV4_ERR_INVALID_ARG = -1, /* null pointer, negative size, inconsistent dims */
  DSV4_ERR_UNSUPPORTED = -2, /* dims outside the supported ranges below */
  DSV4_ERR_MISALIGNED = -3,  /* a plane not 16-byte aligned */
  DSV4_ERR_WORKSPACE = -4,   /* ws smaller than dsv4_workspace_size() */
  DSV4_ERR_CUDA = -5,        /* a kernel launch failed */
  DSV4_ERR_SCRATCH = -6      /* the call needs more scratch than DSV4_STATIC_SCRATCH_BYTES */
};

/* Bits of the device status word (sticky until dsv4_read_status clears them). */
enum {
  DSV4_STATUS_CAPACITY = 1, /* an append would pass `capacity`: that sequence was left unchanged */
  DSV4_STATUS_BAD_INDEX = 2, /* a top-k index outside [-1, n_c) was ignored */
  DSV4_STATUS_TIMEOUT = 4,   /* a bounded wait inside a kernel expired; that kernel's output is incomplete */
  DSV4_STATUS_RANGE = 8      /* attention met a query, key or value of magnitude >= 65504, outside the f16
                                range of its tensor-core operands; that call's output is unreliable */
};

/* Shape of one attention layer's cache. Supported: 16 <= d_nope <= 512 and a
 * multiple of 16; 0 <= d_rope <= 128 and a multiple of 8; 1 <= ratio <= 256;
 * d_nope + d_rope <= 576; 0 <= window <= 4096; idx_dim 0 (no indexer, HCA),
 * 64, 128 or 256; capacity >= 1 and batch * capacity < 2^31. */
typedef struct {
  int32_t batch;      /* B sequences */
  int32_t d_nope;     /* FP8 dims of an entry */
  int32_t d_rope;     /* BF16 (RoPE) dims of an entry; D = d_nope + d_rope */
  int32_t ratio;      /* m tokens pooled into one compressed entry (4 for CSA, 128 for HCA) */
  int32_t window;     /* W raw tokens kept in the sliding-window ring */
  int32_t separate_v; /* 0: one shared entry serves as K and V; 1: separate V planes of the same layout */
  int32_t idx_dim;    /* Di dims of an FP4 indexer key, 0 when the layer has no indexer */
  int32_t capacity;   /* compressed entries each sequence's planes can hold */
} dsv4_layer_desc;

/* Planes of compressed entries [HYB]: entry j of sequence b holds
 * y[j][c] ~= e4m3(nope[b][j][c]) * scale[b][j] for c < d_nope and
 * bf16(rope[b][j][c - d_nope]) for the RoPE dims. */
typedef struct {
  uint8_t* nope;   /* [B][capacity][d_nope] e4m3 codes */
  float* scale;    /* [B][capacity] per-entry fp32 scale = amax(|y_nope|) / 448 */
  uint16_t* rope;  /* [B][capacity][d_rope] bf16 */
} dsv4_kv_planes;

/* All device state of one layer's cache (caller-allocated, zero-initialised
 * before the first append). Token t of sequence b sits in window slot t % W
 * and, while its block is still open, in pending slot t % ratio [CSA]. */
typedef struct {
  dsv4_kv_planes k;     /* keys, or the shared K=V entry */
  dsv4_kv_planes v;     /* values when separate_v, else unused (NULL) */
  uint8_t* idx_codes;   /* [B][capacity][Di/2] e2m1 indexer keys, NULL when idx_dim == 0 */
  uint8_t* idx_scales;  /* [B][capacity][Di/16] e4m3 scales, one per 16 dims */
  uint16_t* win_k;      /* [B][W][D] bf16 raw keys of the last W tokens (ring) */
  uint16_t* win_v;      /* [B][W][D] bf16 raw values (separate_v only) */
  uint16_t* pend_k;     /* [B][ratio][D] bf16 tokens of the open block */
  uint16_t* pend_v;     /* [B][ratio][D] (separate_v only) */
  uint16_t* pend_z;     /* [B][ratio][D] gate logits of the open block */
  uint16_t* pend_u;     /* [B][ratio][Di] indexer-key tokens of the open block */
  uint16_t* pend_zu;    /* [B][ratio][Di] their gate logits */
  int64_t* n_tokens;    /* [B] tokens appended so far */
  int32_t* status;      /* one int32 status word */
} dsv4_cache;

/* Append T tokens to every sequence [HYB], [CSA].
 * For every block [j*m, (j+1)*m) that this call completes, channel by channel:
 *   y[c] = sum_i softmax_i(z[jm+i][c] + b[i][c]) * x[jm+i][c]     (fp32)
 * then y is stored as an FP8 entry (scale = amax/448, codes = e4m3(y/scale),
 * RoPE dims bf16); with an indexer, the u stream is pooled the same way with
 * zu and bu and stored as FP4 (per 16 dims: scale = e4m3(amax/6),
 * codes = e2m1(y/scale)). The last W tokens go to the window ring, the tokens
 * of a still-open block to the pending planes, and n_tokens advances by T.
 *   k, z : [B][T][D] bf16 keys (post-RoPE) and gate logits
 *   v    : [B][T][D] bf16 values, NULL unless separate_v (the same gates apply)
 *   b    : [ratio][D] fp32 position bias
 *   u, zu: [B][T][Di] bf16 indexer-key stream and its gate logits (NULL when idx_dim == 0)
 *   bu   : [ratio][Di] fp32 position bias of the indexer-key pooling
 * A sequence whose entries would pass `capacity` is left unchanged and sets
 * DSV4_STATUS_CAPACITY. T may be 0. */
int dsv4_compress_append(const dsv4_layer_desc* desc, const dsv4_cache* cache, int32_t T,
                         const uint16_t* k, const uint16_t* v, const uint16_t* z, const float* b,
                         const uint16_t* u, const uint16_t* zu, const float* bu, void* stream);

/* Lightning indexer and top-k selection [HYB], [CSA].
 * The query q_idx [B][Hi][Di] (bf16) is quantised to FP4 with the same rule as
 * the keys; for each compressed entry s < n_c = n_tokens[b] / ratio,
 *   I[b][s] = sum_h w[b][h] * max(0, q_h . k_s)      (decoded FP4 values)
 * and topk[b] receives the k entries with the largest I (ties to the lower
 * index) in ascending index order, padded with -1 when n_c < k.
 *   w      : [B][Hi] fp32 head weights
 *   topk   : [B][k] int32 output
 *   scores : [B][capacity] fp32 output of I (entries >= n_c untouched), or NULL
 *   ws     : device workspace of at least dsv4_workspace_size() bytes
 * The contraction runs on the tensor cores (block-scaled FP4 MMA, fp32 accumulate).
 * Supported: 1 <= Hi <= 128, 1 <= k <= 2048, layer with idx_dim > 0. */
int dsv4_index_topk(const dsv4_layer_desc* desc, const dsv4_cache* cache, int32_t Hi,
                    const uint16_t* q_idx, const float* w, int32_t k, int32_t* topk, float* scores,
                    void* ws, size_t ws_bytes, void* stream);

/* CSA attention [HYB], [CSA]: for each head h one softmax over the union of the
 * selected compressed entries and the window tokens (the last min(W, n)):
 *   s_j = sm_scale * q_h . key_j,  out[b][h] = sum_j softmax(s)_j value_j,
 *   lse[b][h] = log sum_j exp(s_j)  (natural log; -inf and out = 0 for an empty set)
 * with key/value of an entry = [e4m3 codes * scale || bf16 rope] and of a
 * window token its raw bf16 row; V = K for a shared entry.
 *   q    : [B][H][D] bf16 query (used exactly)
 *   topk : [B][k] int32 entry indices (-1 = none); duplicates count twice
 *   out  : [B][H][D] fp32;  lse : [B][H] fp32 or NULL
 * k = 0 attends over the window alone (topk is not read and may be NULL): the
 * standard sliding-window layer that follows the CSA / HCA stack ([HCA]).
 * Supported: 1 <= H <= 128, 0 <= k <= 2048. */
int dsv4_csa_decode(const dsv4_layer_desc* desc, const dsv4_cache* cache, int32_t H,
                    const uint16_t* q, float sm_scale, const int32_t* topk, int32_t k,
                    float* out, float* lse, void* ws, size_t ws_bytes, void* stream);

/* HCA attention [HYB], [HCA]: as dsv4_csa_decode over every compressed entry
 * (n_tokens[b] / ratio of them) together with the window tokens. */
int dsv4_hca_decode(const dsv4_layer_desc* desc, const dsv4_cache* cache, int32_t H,
                    const uint16_t* q, float sm_scale, float* out, float* lse,
                    void* ws, size_t ws_bytes, void* stream);

/* Multi-token decode (chunked prefill, speculative decoding) [CSA]: the
 * compressor outputs entries for T new tokens per step, and all T queries of a
 * sequence are served in one call, after their tokens were appended. Query t
 * of sequence b sits at position p = n_tokens[b] - T + t and sees the tokens
 * up to p only: the compressed entries complete by then, n_c(t) = (p + 1) /
 * ratio (its indexer scores and top-k cover those alone: a causal selection),
 * and the window of the min(W, p + 1) raw tokens ending at p. The cache's ring
 * holds only the last W tokens, so the window tokens come from a span of raw
 * rows the caller passes:
 *   span_k, span_v : [B][T + W - 1][D] bf16 keys (values) of the positions
 *                    [n_tokens[b] - T - W + 1, n_tokens[b]); rows of negative
 *                    positions are not read; span_v only when separate_v.
 * Layouts: q_idx [B][T][Hi][Di], w [B][T][Hi], topk [B][T][k] (index_topk
 * output, csa input), scores [B][T][capacity] or NULL; q [B][T][H][D],
 * out [B][T][H][D], lse [B][T][H] or NULL. Same argument rules as the
 * single-token calls, and batch * T <= 65535; workspace:
 * dsv4_workspace_size_multi(). T = 1 with a span of the last W tokens computes
 * what the single-token calls compute. */
int dsv4_index_topk_multi(const dsv4_layer_desc* desc, const dsv4_cache* cache, int32_t T, int32_t Hi,
                          const uint16_t* q_idx, const float* w, int32_t k, int32_t* topk, float* scores,
                          void* ws, size_t ws_bytes, void* stream);
int dsv4_csa_decode_multi(const dsv4_layer_desc* desc, const dsv4_cache* cache, int32_t T, int32_t H,
                          const uint16_t* q, float sm_scale, const int32_t* topk, int32_t k, const uint16_t* span_k,
                          const uint16_t* span_v, float* out, float* lse, void* ws, size_t ws_bytes, void* stream);
int dsv4_hca_decode_multi(const dsv4_layer_desc* desc, const dsv4_cache* cache, int32_t T, int32_t H,
                          const uint16_t* q, float sm_scale, const uint16_t* span_k, const uint16_t* span_v,
                          float* out, float* lse, void* ws, size_t ws_bytes, void* stream);
size_t dsv4_workspace_size_multi(const dsv4_layer_desc* desc, int32_t T, int32_t H, int32_t Hi, int32_t k);

/* dsv4_hca_decode for callers that cannot allocate device memory.
 * The pages describe no such call; it exists for library users. Some callers
 * cannot call cudaMalloc at all: code that runs while a CUDA graph is being
 * captured, engines whose memory is fully planned up front by an allocator
 * that owns the device, or plug-in hosts that forbid allocation on their
 * hot path. This variant takes the same arguments as dsv4_hca_decode minus the
 * workspace: its split partials live in one file-scope device array of
 * DSV4_STATIC_SCRATCH_BYTES that every GPU loading the library holds until the
 * process exits. The caller still passes the cache, query and outputs.
 *   - Returns DSV4_ERR_SCRATCH (and launches nothing) when the call would need
 *     more than DSV4_STATIC_SCRATCH_BYTES (dsv4_workspace_size(desc, H, 0, 0)
 *     gives the need).
 *   - The first call on a device looks up the array's device address there
 *     (with that device current); make that first call before any stream
 *     capture. Later calls only read the cached address.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; the kernels write every scratch word they read, so nothing needs
 *     clearing between calls. Calls whose executions overlap on the GPU (other
 *     streams, other threads) race on the array: order them.
 *   - It allocates and frees nothing (no cudaMalloc, cudaFree or allocating
 *     library routine). */
#define DSV4_STATIC_SCRATCH_BYTES (32u << 20)
int dsv4_hca_decode_static(const dsv4_layer_desc* desc, const dsv4_cache* cache, int32_t H,
                           const uint16_t* q, float sm_scale, float* out, float* lse, void* stream);

/* Bytes of device workspace the calls above need for this layer with H query
 * heads, Hi indexer heads and top-k k (0 when the arguments are invalid). */
size_t dsv4_workspace_size(const dsv4_layer_desc* desc, int32_t H, int32_t Hi, int32_t k);

/* How a decode call of this layer splits its work (the pages describe no such
 * call: it exposes the launch plan for tests and capacity planning). k is the
 * top-k width of a dsv4_csa_decode call (0: its window-only form), or -1 for
 * dsv4_hca_decode. Writes plan[0..5] = {tensor-core path (1) or CUDA-core path
 * (0), splits per (sequence, head group), rows per tile (tensor-core path) or
 * rows per split (CUDA-core path), tiles per split, head groups of 64,
 * streaming multiprocessors planned for}. Host only; launches nothing. */
int dsv4_decode_plan(const dsv4_layer_desc* desc, int32_t H, int32_t k, int32_t* plan);

/* The streams dsv4_compress_append pools, projected from hidden states with
 * RoPE, on the tensor cores [HYB] (the pooling is learned: its inputs are
 * projections of the token's hidden state), [ROPE] (positions enter through
 * RoPE).
 *   hidden  [B][T][d_model] bf16: T new tokens of every sequence;
 *   weight  [2 D + 2 Di][d_model] bf16: the rows of the x, z, u and zu
 *           projections in that order (D = d_nope + d_rope, Di = idx_dim);
 *   x, z    [B][T][D] bf16 outputs; u, zu [B][T][Di] bf16 (NULL when Di = 0).
 * Per token at position p = n_tokens[b] + t (the cache's count before the
 * append of these tokens, so call this first): y = W . h in fp32 (bf16
 * products, fp32 accumulation), then RoPE on the trailing d_rope dims of x
 * and the trailing min(d_rope, Di) dims of u: pair (2i, 2i + 1) of those dims
 * turns by p * rope_base^(-2i/d) (d the number of rotated dims), and every
 * value is rounded once to bf16. Positions are exact below 2^24.
 * Requirements: shared K = V (separate_v = 0), d_model a multiple of 64,
 * d_nope, D and Di multiples of 32, d_rope <= 64, rope_base > 1
 * (DSV4_ERR_UNSUPPORTED / DSV4_ERR_INVALID_ARG otherwise). T may be 0. */
int dsv4_project_streams(const dsv4_layer_desc* d, const dsv4_cache* c, int32_t T, int32_t d_model,
                         const uint16_t* hidden, const uint16_t* weight, float rope_base, uint16_t* x, uint16_t* z,
                         uint16_t* u, uint16_t* zu, void* stream);

/* Test hook of the failure path (the pages describe no such call). While on
 * != 0, every tensor-core attention kernel launched by the decode calls makes
 * its MMA-issuing thread first wait on a barrier that nothing arrives on: the
 * bounded wait runs out after 50 ms, every role of the kernel leaves its loop
 * (copies and MMAs in flight drained), the call's output is not computed, and
 * DSV4_STATUS_TIMEOUT is raised in the cache's status word. Affects the current
 * device only; call with 0 to restore normal operation. For tests. */
int dsv4_debug_force_timeout(int32_t on);

/* Waits for `stream`, then returns the cache's status bits (>= 0) and clears
 * them; a negative DSV4_ERR_* on failure. */
int dsv4_read_status(const dsv4_cache* cache, void* stream);

/* The quantisation step of an append on rows pooled elsewhere [HYB]:
 * y [rows][d_nope + d_rope] fp32 -> nope [rows][d_nope] e4m3, scale [rows],
 * rope [rows][d_rope] bf16, with the same rule and rounding as
 * dsv4_compress_append. Alignment: y, scale 4 bytes; nope, rope 2 bytes (so that
 * one sequence's slice of a cache plane can be filled directly). */
int dsv4_quantize_kv_rows(const float* y, int64_t rows, int32_t d_nope, int32_t d_rope,
                          uint8_t* nope, float* scale, uint16_t* rope, void* stream);

/* FP4 quantisation of rows [HYB]: y [rows][cols] fp32 (cols a multiple of 32)
 * -> codes [rows][cols/2] e2m1, scales [rows][cols/16] e4m3. Alignment: y 16 bytes,
 * codes 4 bytes, scales none. */
int dsv4_quantize_fp4_rows(const float* y, int64_t rows, int32_t cols, uint8_t* codes,
                           uint8_t* scales, void* stream);

/* The pooling step of an append on complete blocks [HYB]:
 * x, z [blocks * ratio][dim] bf16, b [ratio][dim] fp32 -> y [blocks][dim] fp32,
 * with the arithmetic of dsv4_compress_append. dim a multiple of 8, at most 4096. */
int dsv4_pool_rows(const uint16_t* x, const uint16_t* z, const float* b, int64_t blocks,
                   int32_t ratio, int32_t dim, float* y, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSV4_H */
