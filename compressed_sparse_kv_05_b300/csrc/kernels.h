// Internal declarations shared by the libdsv4 translation units: argument
// blocks handed to the kernels and the kernels themselves.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsv4 {

// Several queries per sequence (multi-token decode): virtual sequence v = b * T
// + t is query t of sequence b, at position n_tokens[b] - T + t; it reads
// sequence b's cache planes and sees the tokens up to its own position.
// T = 1 is single-token decode (v = b).
__device__ __forceinline__ int64_t vseq_tokens(const int64_t* n_tokens, int v, int T) {
  const int64_t n = n_tokens[v / T] - (T - 1 - v % T);
  return n > 0 ? n : 0;
}

struct AppendArgs {
  int T, ratio, window, capacity, d_nope, d_rope, idx_dim, separate_v;
  int ctas_k;              // pool_chunk_kernel: CTAs of the key (and value) stream, then
  int ctas_u;              //   CTAs of the indexer-key stream, then CTAs copying window rows (kWinRowsPerCta each)
  int bpc_k, bpc_u;        // blocks per CTA of each stream
  const uint16_t *k, *v, *z, *u, *zu;
  const float *bias, *bias_u;
  uint8_t* k_nope;
  float* k_scale;
  uint16_t* k_rope;
  uint8_t* v_nope;
  float* v_scale;
  uint16_t* v_rope;
  uint8_t *idx_codes, *idx_scales;
  uint16_t *win_k, *win_v, *pend_k, *pend_v, *pend_z, *pend_u, *pend_zu;
  int64_t* n_tokens;
  int32_t* status;
};

// How one compressed block's pooling is shared out, the same in every kernel
// that pools (so a block's pooled bits never depend on how its tokens
// arrived): a team of G * cg threads, cg = C / 8 groups of 8 channels, G
// groups of tpg consecutive tokens (the last may be shorter), at most 512
// threads.
struct PoolShape {
  int cg, G, tpg;
};
__host__ __device__ inline PoolShape pool_shape(int m, int C) {
  PoolShape p;
  p.cg = C / 8;
  int G = (m + 7) / 8;
  const int gmax = p.cg <= 512 ? 512 / p.cg : 1;
  if (G > gmax) G = gmax;
  if (G < 1) G = 1;
  p.G = G;
  p.tpg = (m + G - 1) / G;
  return p;
}
// channels a thread takes when a 64-channel slice of a block with G token
// groups is pooled from shared memory (pool_cluster_kernel): 64 / CPT x G
// threads, at most 256
__host__ __device__ inline int slice_cpt(int G) { return G <= 8 ? 2 : (G <= 16 ? 4 : 8); }
// shared-memory floats a team needs to combine its token groups (0 when G == 1)
__host__ __device__ inline int pool_part_floats(PoolShape p, bool two) {
  return p.G > 1 ? p.G * p.cg * (two ? 24 : 16) : 0;
}

constexpr int kWinRowsPerCta = 16;
__global__ void pool_chunk_kernel(AppendArgs a);
__global__ void pool_cluster_kernel(AppendArgs a);
__global__ void append_tail_kernel(AppendArgs a);
__global__ void append_one_kernel(AppendArgs a);
__global__ void quant_kv_rows_kernel(const float* y, int64_t rows, int d_nope, int d_rope, uint8_t* nope,
                                     float* scale, uint16_t* rope);
__global__ void quant_fp4_rows_kernel(const float* y, int64_t rows, int cols, uint8_t* codes, uint8_t* scales);
__global__ void pool_rows_kernel(const uint16_t* x, const uint16_t* z, const float* bias, int ratio, int dim,
                                 float* y);

// ---- indexer + top-k
// Per-sequence counter words of the top-k: [0] blocks above the threshold bin,
// [1] candidates in it, [2] finished selection CTAs; the rest unused.
constexpr int kCntWords = 8;
struct IndexArgs {
  int B, Hi, N, Di, k, capacity, ratio;
  int T;                   // queries per sequence: B counts B_seq * T virtual sequences (see vseq_tokens)
  const uint16_t* q_idx;   // [B][Hi][Di] bf16
  const float* w;          // [B][Hi]
  const int64_t* n_tokens;
  uint8_t* q_codes;        // [B][N][Di/2] FP4 query, heads padded to N with zeros (workspace)
  uint8_t* q_scales;       // [B][N][Di/16]
  float* scores;           // [B][capacity]
  int32_t* topk;           // [B][k]
  uint32_t* hist1;         // [B][4096] histogram of score-key bits 31..20 (filled while scoring)
  uint32_t* hist2;         // [B][4096] histogram of key bits 19..8 inside the threshold bin
  uint32_t* cnt;           // [B][kCntWords] (see kCntWords)
  int32_t* above;          // [B][k] blocks above the threshold bin
  uint64_t* cand;          // [B][capacity] (key << 32 | index) of the blocks in the threshold bin
  int32_t* status;         // the cache's status word
};
__global__ void quant_query_fp4_kernel(IndexArgs a);
__global__ void topk_select_kernel(IndexArgs a);
// Projection of the compressor's streams from hidden states with RoPE (project.cu).
struct ProjArgs {
  int M, N, K;                 // token rows (B * T), output columns (2 D + 2 Di), hidden size
  int T;                       // tokens per sequence: row r is token r % T of sequence r / T
  int d_nope, d_rope, Di, ur;  // ur = min(d_rope, Di) rotated dims of u
  int bn, tiles_n, tiles;      // tile width and tile counts, set by launch_project
  const int64_t* n_tokens;     // [B] tokens before this call: positions n_tokens[b] + t
  uint16_t *x, *z, *u, *zu;    // [M][D], [M][D], [M][Di], [M][Di] bf16
  int32_t* status;
  float rx_hi[32], rx_lo[32];  // theta_i / pi of x's rotated dims as float pairs (set by launch_project)
  float ru_hi[32], ru_lo[32];  // and of u's
};
int launch_project(ProjArgs a, const void* hidden, const void* weight, double rope_base, int sms, cudaStream_t st);

// Top-k launch: the cluster kernel (topk_cluster_kernel) when topk_plan finds
// a cluster size and per-thread score count for the capacity, else the
// global-atomic kernel with sel_ctas CTAs per sequence.
int topk_plan(int B, int capacity, int sms, int* cluster_ctas, int* per_thread);
int launch_topk_select(const IndexArgs& a, int sel_ctas, int sms, cudaStream_t st);

struct IndexTcArgs {
  int B, N, Di, capacity, ratio, ctas_per_seq, k;
  int T;                       // queries per sequence (B counts virtual sequences)
  uint32_t tmem_cols;
  const int64_t* n_tokens;
  const uint8_t* idx_codes;    // [B][capacity][Di/2] (read through the tensor map; its address for L2 prefetches)
  const uint8_t* idx_scales;   // [B][capacity][Di/16]
  const uint8_t* q_scales;     // [B][N][Di/16]
  const float* w;              // [B][Hi] head weights (the caller's input)
  int Hi;
  float* scores;               // [B][capacity]
  uint32_t* hist1;             // [B][4096]
  uint32_t* cnt;               // [B][kCntWords]
  int32_t* status;
};
// tcgen05 block-scaled FP4 scores; key_codes [B][capacity][Di/2], q_codes [B][N][Di/2]
int launch_index_scores_tc(const IndexTcArgs& a, const uint8_t* key_codes, const uint8_t* q_codes, cudaStream_t st);

// ---- attention
struct AttnArgs {
  int B, H, D, Dv, d_nope, d_rope, ratio, window, capacity, separate_v;
  int T;                   // queries per sequence: B counts B_seq * T virtual sequences (see vseq_tokens)
  int span;                // 0: window tokens from the cache's ring (win_k: [B_seq][W][D]); else rows per
                           // sequence of a span of recent raw tokens (win_k: [B_seq][span][D], the tokens at
                           // positions [n - span, n) of a sequence holding n tokens)
  int n_sel;               // top-k width (CSA), 0 for HCA (every entry), -1 for none (window only)
  int splits, rows_per_split;
  int tile_rows;           // tensor-core kernel: rows per tile (32, 64 or 128)
  int tiles_per_split;     // tensor-core kernel: tiles per CTA
  int tma;                 // tensor-core kernel: the compressed rows arrive by TMA boxes (AttnMaps valid)
  float sm_scale;
  const uint16_t* q;
  const int32_t* topk;
  const uint8_t *k_nope, *v_nope;
  const float *k_scale, *v_scale;
  const uint16_t *k_rope, *v_rope, *win_k, *win_v;
  const int64_t* n_tokens;
  int32_t* status;
  float* part_o;           // [B][H][splits][Dv] fp32 (CUDA-core kernel); f16 [B][splits][hg][D][64], granules swizzled (tensor-core)
  float* part_lse;         // [B][H][splits] natural-log sum of each split's softmax weights
  float* part_lsev;        // [B][H][splits] tensor-core kernel: natural log of the scale of its normalised partial
  float* out;              // [B][H][Dv]
  float* lse;              // [B][H] or null
};
// Tensor maps of the contiguous compressed rows (HCA) for the tensor-core
// kernel: boxes of tile_rows rows x 128 code bytes, x the last chunk's code
// bytes, and x all RoPE bytes of a row.
struct AttnMaps {
  CUtensorMap nope, nope_tail, rope;
};
// launches the split kernel over (splits, B, head_groups) and the merge; returns a DSV4 status
int launch_attention(const AttnArgs& a, int head_groups, cudaStream_t st);
// the tensor-core split kernel (tiles of up to 128 rows, up to 64 heads per CTA) and the merge
bool attention_tc_supported(int H, int d_nope, int d_rope, int separate_v);
// test hook of the tensor-core attention: its MMA thread's first wait runs out (see attention_tc.cu)
int attention_force_timeout(int on);
// whether the tensor-core kernel can take the compressed rows of this shape by TMA boxes
bool attention_tc_tma_shape(int d_nope, int d_rope, int separate_v);
int launch_attention_tc(const AttnArgs& a, int head_groups, cudaStream_t st);
int launch_attention_merge(const AttnArgs& a, cudaStream_t st);
// merge of the tensor-core kernel's f16 partials ([B][splits][head groups][D][64])
int launch_attention_merge_tc(const AttnArgs& a, int head_groups, cudaStream_t st);
// 2D tensor map over `rows` rows of `row_bytes` bytes (uint8, no swizzle), box
// of box_bytes x box_rows; false if the driver's encoder is unavailable or refuses
bool encode_u8_rows(CUtensorMap* map, const void* base, int64_t rows, int row_bytes, int box_bytes, int box_rows);

}  // namespace dsv4
