// CSA / HCA decode attention on the 5th-generation tensor cores (tcgen05
// kind::f16, fp32 accumulators in tensor memory).
//
// vibecoco.ai, "DeepSeek V4 agent architecture", section
// "混合注意力：两种压缩，交替使用": CSA attends over the top-k compressed blocks
// plus a sliding window of recent raw tokens, HCA densely over every
// compressed entry plus the window; every query head shares the one KV head.
// pnsm.cn, "DeepSeek V4 架构深度解析…", section 2.1 "CSA：压缩稀疏注意力": the
// window and the compressed KV feed one attention (one softmax over the union).
//
// All query heads read the same rows, so a decode step is a pair of dense
// contractions per tile of up to 128 rows:
//   X   [128 rows][D]  f16: each row's dequantised key (code * scale || rope, or
//                      the raw window token); it is also the value row when K = V
//   S^T [128][64]      = X . Q^T             (M = 128 rows, N = 64 heads, K = D)
//   P   [128][64]      = exp2(S^T * c - m)   (f16, the running max m per head)
//   O^T [D][64]       += X^T . P             (M = 128 dims per block, N = 64, K = rows)
// X is written once per tile in the 128-byte-swizzled layout that serves as a
// K-major operand for the first product and as an MN-major operand for the
// second; S^T and O^T live in tensor memory (lane = row / dim, column = head).
//
// A sequence's rows are cut into tiles of R = 32, 64 or 128 rows (the host
// picks the largest R that still fills the GPU): first the compressed rows
// (the top-k list for CSA, every entry for HCA), then the window tokens; a tile
// never mixes the two. Each CTA takes a run of consecutive tiles (a split).
// X is staged chunk by chunk, a chunk being 128 dims of every row of the tile:
// the raw bytes land in the chunk's own region of X and are dequantised there.
//
// CTA roles (512 threads, one CTA per SM for D = 512):
//   warp 0      allocates tensor memory; one lane issues every MMA;
//   warp 1      one lane streams the compressed rows of HCA tiles with TMA
//               boxes (contiguous rows); the others prefetch later tiles into L2;
//   warps 2-15  (448 workers) copy gathered rows (CSA, and every window token)
//               with cp.async, convert the query, and dequantise every chunk in
//               place (see "row exponents" below).
//               Warps 4-7 and 12-15 (two per 32-lane quarter of tensor memory)
//               also turn S^T into P (see below). After the last tile they
//               normalise O^T and store this split's partial output as f16
//               (rows of 64 heads per dim, 16-byte granules swizzled by dim).
// Splits are merged by attn_merge_tc_kernel (attention.cu).
//
// Row multipliers. Every row j of a tile is held in X as a normalised f16 row
// X_j = key_j / mu_j, with a positive fp32 multiplier mu_j per row:
//   entry   mu_j = 256 * scale_j: the codes become code * 2^-8, exactly (the
//           hardware e4m3 -> f16 conversion is exact, the multiply by 2^-8
//           too), and the RoPE dims rope / mu_j (rounded once);
//   window  mu_j = 2^L_j, L_j the binade of the row's largest |value| over all
//           D dims (the row lands in [1, 2) at its largest element).
// So f16 holds every row to 11 significant bits whatever the entry's scale or
// the token's magnitude, and an entry's FP8 dims exactly. The scores take the
// multiplier back in fp32:
//   s_jh = (X_j . q_h) * mu_j * sm_scale * log2(e)               (log2 domain)
// and the normaliser of head h is l_h = sum_j 2^(s_jh - m_h) with a running
// max m_h. The value side keeps its own running max M_h of s_jh + L'_j (L'_j
// the binade of mu'_j, the multiplier of row j's value row: mu_j itself when
// K = V):
//   P_jh = 2^(s_jh - M_h) mu'_j = p_jh * (mu'_j / 2^T) * 2^(T + m_h - M_h),
//   O_h = sum_j P_jh X'_j,
// with p_jh = 2^(s_jh - m_h), T the largest L'_j of the tile: a factor of the
// row (< 2) and a power of two of the head. Both maxima are integers that
// move only when a tile exceeds them by more than 2^8 (then l, resp. O^T, is
// rescaled by an exact power of two), so p <= 256 and P < 512. The split's
// partial output is stored normalised by l'_h = sum_j P_jh (a convex
// combination of normalised rows, so it fits f16) with two natural-log sums:
// lse = ln(2^m_h l_h) and lse' = ln(2^M_h l'_h); the merge weighs each
// split's partial by exp(lse' - max lse) and divides by sum exp(lse - max lse).
//
// Precision: the RoPE dims and window values in X, P and the split partials
// are rounded to f16 (relative error <= 2^-11 each); the FP8 dims are exact;
// the bf16 query converts to f16 exactly for |q| in [2^-14, 65504]; products,
// sums and multipliers are fp32. A query element of
// magnitude >= 65504, or RoPE dims more than 2^15 times an entry's largest FP8
// value, do not fit the f16 operands and raise DSV4_STATUS_RANGE. The two
// e4m3 NaN codes (never written by the quantiser) decode to NaN, as the format
// defines them.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace dsv4 {

namespace {

constexpr int kRows = 128;                     // MMA M; the most rows a tile holds
constexpr int kHeads = 64;                     // heads per CTA (MMA N), zero-padded
constexpr int kThreads = 512;
constexpr int kWorkers = 14 * 32;              // warps 2-15
constexpr int kSoftThreads = 8 * 32;           // warps 4-7 and 12-15
constexpr int kGroups = kRows * 16;            // 8-dim groups of one 128-dim chunk
constexpr int kItems = (kGroups + kWorkers - 1) / kWorkers;
constexpr int kQItems = (kHeads * 64 + kWorkers - 1) / kWorkers;   // 8-dim query groups (D <= 512)
constexpr int kAtomBytes = kRows * 128;        // 128 rows x 64 dims f16
constexpr int kChunkBytes = 2 * kAtomBytes;    // 128 rows x 128 dims f16
constexpr int kQAtomBytes = kHeads * 128;      // 64 heads x 64 dims f16
constexpr int kPBytes = kRows * kHeads * 2;
constexpr int kMaxChunks = 4;                  // D <= 512
constexpr int kMaxTiles = 8;                   // tiles per CTA (the host plan keeps to it)
constexpr int kBarWork = 1, kBarSoft = 2;      // named barriers (0 is __syncthreads)
constexpr float kRescale = 8.f;                // lazy-rescale threshold (log2 units)
constexpr float kF16Max = 65504.f;

// Test hook (dsv4_debug_force_timeout): when set, the MMA thread of every
// attention CTA first waits on a barrier that nothing arrives on, so that its
// bounded wait runs out after kForcedWaitNs and the kernel takes its timeout
// path (abort flag, every role leaves its loop, copies and MMAs drained,
// DSV4_STATUS_TIMEOUT raised). Never set outside tests.
__device__ int g_force_timeout = 0;
constexpr uint64_t kForcedWaitNs = 50000000ull;   // 50 ms

struct TcTail {
  uint64_t xland[kMaxChunks], xfull[kMaxChunks], xfree[kMaxChunks], sfull, pfull, qready, drain, never;
  uint32_t taddr;
  int abort;
  // the per-row arrays are 16-byte aligned: the scales of a tile arrive by bulk copies
  alignas(16) int32_t src[kMaxTiles * kRows];   // row sources of every tile of the split (see row_source), 128 per tile
  alignas(16) uint32_t sk[kMaxTiles * kRows];   // key (or shared entry) scale of every row: raw fp32 until the
                                                // tile's first chunk turns it into f_j as f16x2 (0 for others)
  alignas(16) uint32_t sv[kMaxTiles * kRows];   // the same for the value scale (separate V); with a shared
                                                // entry, the row multipliers instead (see row_muls)
  int32_t texv[kMaxTiles];            // T: the largest value-row binade of each tile (kNoExp: none yet)
  int32_t texn[kMaxTiles];            // the smallest one (-kNoExp: none yet)
  alignas(16) float m_used[kHeads];   // normaliser running max per head, log2 domain, an integer (read as float4)
  alignas(16) float mv_used[kHeads];  // value-side running max per head, an integer
  alignas(16) float alpha[kHeads];    // rescale of l (then 1 / l' in the epilogue)
  alignas(16) float alphav[kHeads];   // rescale of O^T
  alignas(16) float phi[2][kHeads];   // 2^(T + m - M) per head for tiles of even / odd index
  float lsum[kHeads];
  float lvsum[kHeads];
  float red[4][kHeads];
  float redv[4][kHeads];
};

constexpr int kNoExp = -1000;   // tile exponent before any row of the tile was seen

// Reciprocal row multipliers 1 / mu_j of every row of the split (128 per
// tile, fp32): the key rows', then (separate V) the value rows'. With a shared
// entry they live in the unused value-scale array; with separate V they follow
// the tail in shared memory.
template <bool SEP>
DSV4_DEV float* row_muls(TcTail* t) {
  return SEP ? reinterpret_cast<float*>(t + 1) : reinterpret_cast<float*>(t->sv);
}
constexpr int kMulsPerSplit = kMaxTiles * kRows;
// 2^e as fp32 for an integer e in [-126, 127] (exact).
DSV4_DEV float pow2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// The binade of x > 0 (floor(log2 x)) clamped to [-126, hi]; 0 for x == 0.
DSV4_DEV int binade(float x, int hi = 126) {
  const int e = static_cast<int>((__float_as_uint(x) >> 23) & 0xFFu) - 127;
  return x > 0.f ? (e < -126 ? -126 : (e > hi ? hi : e)) : 0;
}

// 2^(a - b) for integer-valued a <= b (exact); 0 when a = -inf, 1 when both are -inf.
DSV4_DEV float pow2_diff(float a, float b) {
  if (b == -INFINITY) return 1.f;
  if (a == -INFINITY) return 0.f;
  const float k = a - b;
  return k < -126.f ? 0.f : pow2i(static_cast<int>(k));
}

// 2^k for any integer k, clamped to the normal fp32 range [2^-126, 2^127]
// (below it a product with a weight <= 256 lies far below f16's range).
DSV4_DEV float pow2_clamped(int k) { return pow2i(k < -126 ? -126 : (k > 127 ? 127 : k)); }

DSV4_DEV uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

DSV4_DEV uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two e4m3 codes (the low and high byte of `two`) times the f16x2 `sc`
// (= scale * 2^8 in both halves): the hardware conversion is exact, the
// multiply by 2^-8 is exact too (it keeps every e4m3 value, subnormals
// included, within f16), and the last multiply rounds once.
DSV4_DEV uint32_t e4m3x2_to_f16x2_scaled(uint16_t two, uint32_t sc) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
  return hmul2(hmul2(h, 0x1C001C00u), sc);   // 0x1C00 = f16 2^-8
}

DSV4_DEV uint32_t bf16x2_to_f16x2(uint32_t w, float& mx) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
  mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
  return f32x2_to_f16x2(lo, hi);
}

DSV4_DEV uint4 bf16x8_to_f16x8(uint4 w, float& mx) {
  return make_uint4(bf16x2_to_f16x2(w.x, mx), bf16x2_to_f16x2(w.y, mx), bf16x2_to_f16x2(w.z, mx),
                    bf16x2_to_f16x2(w.w, mx));
}

// bf16 pair times a power of two (exact in fp32), then rounded to f16 once.
DSV4_DEV uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float sc, float& mx) {
  const float lo = __uint_as_float(w << 16) * sc, hi = __uint_as_float(w & 0xFFFF0000u) * sc;
  mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
  return f32x2_to_f16x2(lo, hi);
}

DSV4_DEV uint4 bf16x8_to_f16x8_scaled(uint4 w, float sc, float& mx) {
  return make_uint4(bf16x2_to_f16x2_scaled(w.x, sc, mx), bf16x2_to_f16x2_scaled(w.y, sc, mx),
                    bf16x2_to_f16x2_scaled(w.z, sc, mx), bf16x2_to_f16x2_scaled(w.w, sc, mx));
}

// Largest |bf16| of 8 values, as the 15 magnitude bits of a bf16.
DSV4_DEV uint32_t bf16x8_absmax_bits(uint4 w) {
  const uint32_t m = 0x7FFF7FFFu;
  const uint32_t a = __vmaxu2(__vmaxu2(w.x & m, w.y & m), __vmaxu2(w.z & m, w.w & m));
  const uint32_t lo = a & 0xFFFFu, hi = a >> 16;
  return lo > hi ? lo : hi;
}

DSV4_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Rows of sequence b: n_main compressed rows (the top-k list for CSA, every
// entry for HCA), then n_win window tokens, oldest first.
struct RowSpace {
  int64_t n_tok, n_c, n_win, n_main;
  int mt, wt;   // tiles of compressed rows, tiles of window rows
};

DSV4_DEV RowSpace row_space(const AttnArgs& a, int b) {
  RowSpace s;
  s.n_tok = vseq_tokens(a.n_tokens, b, a.T);
  s.n_c = s.n_tok / a.ratio < a.capacity ? s.n_tok / a.ratio : a.capacity;
  s.n_win = s.n_tok < a.window ? s.n_tok : a.window;
  s.n_main = a.n_sel > 0 ? a.n_sel : (a.n_sel < 0 ? 0 : s.n_c);
  s.mt = static_cast<int>((s.n_main + a.tile_rows - 1) / a.tile_rows);
  s.wt = static_cast<int>((s.n_win + a.tile_rows - 1) / a.tile_rows);
  return s;
}

// Tile i of a sequence: rows [r0, r0 + cnt) of the compressed rows, or of the
// window tokens when win.
struct Tile {
  bool win;
  int64_t r0;
  int cnt;
};

DSV4_DEV Tile tile_at(const AttnArgs& a, const RowSpace& s, int i) {
  Tile t;
  t.win = i >= s.mt;
  t.r0 = static_cast<int64_t>(t.win ? i - s.mt : i) * a.tile_rows;
  const int64_t left = (t.win ? s.n_win : s.n_main) - t.r0;
  t.cnt = static_cast<int>(left < a.tile_rows ? left : a.tile_rows);
  return t;
}

// Source of row j of tile t of virtual sequence b: >= 0 entry index into the
// planes (b_seq * capacity + e), -1 no row (past the tile, a -1 top-k slot or
// an invalid index), <= -2 a row of the window source (-2 - row): of the ring
// (b_seq * W + position % W) or of the span (b_seq * span + position - the
// span's first position).
DSV4_DEV int32_t row_source(const AttnArgs& a, const RowSpace& s, int b, const Tile& t, int j) {
  if (j >= t.cnt) return -1;
  const int64_t r = t.r0 + j;
  const int64_t bs = b / a.T;
  if (!t.win) {
    const int64_t e = a.n_sel > 0 ? static_cast<int64_t>(a.topk[static_cast<int64_t>(b) * a.n_sel + r]) : r;
    if (e < -1 || e >= s.n_c) {
      atomicOr(a.status, DSV4_STATUS_BAD_INDEX);
      return -1;
    }
    if (e < 0) return -1;
    return static_cast<int32_t>(bs * a.capacity + e);
  }
  const int64_t pos = s.n_tok - s.n_win + r;
  if (a.span == 0) return static_cast<int32_t>(-2 - (bs * a.window + pos % a.window));
  return static_cast<int32_t>(-2 - (bs * a.span + pos - (a.n_tokens[bs] - a.span)));
}

DSV4_DEV void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
DSV4_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most n of this thread's committed groups are pending (n < 4)
DSV4_DEV void cp_async_wait(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
  }
}

// Dims [128c, 128c + 128) of an entry row: nn FP8 codes, then 128 - nn RoPE
// dims (bf16) starting at RoPE element e0. Raw bytes of row j in the chunk's
// region: codes at j * nn, RoPE at rope_off + j * rb (rope_off = 128 * nn, a
// multiple of 128 bytes as a TMA destination needs). A window row's 128 bf16
// values sit at j * 256.
struct ChunkSplit {
  int nn, e0, rb, rope_off;
};
DSV4_DEV ChunkSplit chunk_split(const AttnArgs& a, int c) {
  int nn = a.d_nope - c * 128;
  nn = nn < 0 ? 0 : (nn > 128 ? 128 : nn);
  return ChunkSplit{nn, c * 128 + nn - a.d_nope, 2 * (128 - nn), 128 * nn};
}

// Issue the cp.async copies of chunk c of a tile (row sources `src`, rc rows)
// into the chunk region xc; rows without a source get nothing.
DSV4_DEV void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}

DSV4_DEV void issue_chunk(const AttnArgs& a, int b, bool win, const int32_t* src, int c, int rc, const uint8_t* nope,
                          const uint16_t* rope, const float* scale, const uint16_t* wbuf, unsigned char* xc,
                          uint32_t* sk, int wtid) {
  const ChunkSplit cs = chunk_split(a, c);
  const int ng = cs.nn / 16, nr = cs.rb / 16;
  // with the first chunk, every row's scale (raw fp32, turned into its f16x2
  // multiplier when the chunk converts)
  if (c == 0 && !win && wtid < rc && src[wtid] >= 0) cp_async4(sk + wtid, scale + src[wtid]);
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int i = wtid + it * kWorkers;
    if (i < rc * 16) {
      const int j = i >> 4, g = i & 15;
      const int32_t sr = src[j];
      if (!win && sr >= 0) {
        if (g < ng)
          cp_async16(xc + j * cs.nn + 16 * g, nope + static_cast<int64_t>(sr) * a.d_nope + c * 128 + 16 * g);
        else if (g < ng + nr)
          cp_async16(xc + cs.rope_off + j * cs.rb + 16 * (g - ng),
                     rope + static_cast<int64_t>(sr) * a.d_rope + cs.e0 + 8 * (g - ng));
      } else if (win && sr <= -2) {
        cp_async16(xc + j * 256 + 16 * g, wbuf + static_cast<int64_t>(-2 - sr) * a.D + c * 128 + 8 * g);
      }
    }
  }
}

// Item it of worker wtid in chunk c: row j and 8-dim group g. With 64 code
// dims (the chunk where the RoPE dims start in the 448 + 64 layout) each
// aligned run of 32 items holds only code groups or only RoPE groups (four
// rows each), so every warp takes one kind; otherwise 16 groups per row.
DSV4_DEV void chunk_item(int nn, int i, int& j, int& g) {
  if (nn == 64) {
    const int q = i >> 5, l = i & 31;
    j = ((q >> 1) << 2) + (l >> 3);
    g = ((q & 1) << 3) + (l & 7);
  } else {
    j = i >> 4;
    g = i & 15;
  }
}

DSV4_DEV uint4 codes8_to_f16x8(uint2 w, uint32_t s2) {
  return make_uint4(e4m3x2_to_f16x2_scaled(static_cast<uint16_t>(w.x), s2),
                    e4m3x2_to_f16x2_scaled(static_cast<uint16_t>(w.x >> 16), s2),
                    e4m3x2_to_f16x2_scaled(static_cast<uint16_t>(w.y), s2),
                    e4m3x2_to_f16x2_scaled(static_cast<uint16_t>(w.y >> 16), s2));
}

DSV4_DEV uint32_t f16x2_of(float x) {
  uint32_t s2;
  asm("{\n.reg .b16 t;\ncvt.rn.f16.f32 t, %1;\nmov.b32 %0, {t, t};\n}" : "=r"(s2) : "f"(x));
  return s2;
}

DSV4_DEV void store_group(unsigned char* xc, int j, int g, uint4 h) {
  const int atom = g >> 3, gg = g & 7;
  *reinterpret_cast<uint4*>(xc + atom * kAtomBytes + j * 128 + ((gg ^ (j & 7)) << 4)) = h;
}

// The row multipliers of a compressed tile from its rows' raw scales (landed
// with its first chunk; row wtid's by worker wtid): mu_j = 256 * scale_j, at
// least 2^-118 (so that 1 / mu_j stays finite); 1 for a zero scale. Worker
// wtid turns row wtid's raw scale in place into the f16x2 multiplier of its
// codes, 256 * scale_j / mu_j (1 unless mu_j was raised), and stores 1 / mu_j
// in rinv. With tmax, the tile's largest (smallest) binade of mu_j over rows
// with a source is folded into *tmax (*tmin). Called by every worker (whole warps: the
// reduction needs them), before the worker barrier that precedes the first
// chunk's conversion.
DSV4_DEV void scale_multipliers(const int32_t* src, uint32_t* raw, int rc, int wtid, float* rinv, int32_t* tmax,
                                  int32_t* tmin) {
  int e = kNoExp, f = -kNoExp;
  if (wtid < rc) {
    const float scl = __uint_as_float(raw[wtid]);
    const float m = scl > 0.f ? fmaxf(256.f * scl, 0x1p-118f) : 1.f;
    const float r = __frcp_rn(m);
    raw[wtid] = f16x2_of(256.f * scl * r);
    rinv[wtid] = r;
    if (src[wtid] >= 0) e = f = binade(m);
  }
  if (tmax) {
    e = __reduce_max_sync(0xffffffffu, e);
    f = __reduce_min_sync(0xffffffffu, f);
    if ((wtid & 31) == 0 && e != kNoExp) {
      atomicMax(tmax, e);
      atomicMin(tmin, f);
    }
  }
}

// The row multipliers of a window tile whose chunks have all landed (raw
// bf16, row j's 128 values of chunk c at chunk c's region + 256 j), stored as
// their reciprocals in rinv: mu_j = 2^L_j with
// L_j the binade of the row's largest |value| over the nch chunks; with tmax,
// the tile's largest (smallest) L_j over rows that hold a token is folded
// into *tmax (*tmin).
// The 16 items of a row sit in 16 consecutive workers of one warp (kWorkers is
// a multiple of 32), which combine their maxima by shuffles. Called by every
// worker (whole warps), between the barrier that follows the last copies and
// the one that precedes the first chunk's conversion.
DSV4_DEV void window_multipliers(const unsigned char* x, const int32_t* src, int nch, int rc, int wtid, float* rinv,
                                   int32_t* tmax, int32_t* tmin) {
  int tm = kNoExp, tn = -kNoExp;
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int i = wtid + it * kWorkers;
    const int j = i >> 4, g = i & 15;
    uint32_t m = 0;
    if (i < rc * 16)
      for (int c = 0; c < nch; ++c) {
        const uint32_t v = bf16x8_absmax_bits(*reinterpret_cast<const uint4*>(x + c * kChunkBytes + j * 256 + 16 * g));
        m = v > m ? v : m;
      }
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const uint32_t v = __shfl_xor_sync(0xffffffffu, m, o);
      m = v > m ? v : m;
    }
    if (g == 0 && i < rc * 16) {
      const int L = binade(__uint_as_float(m << 16));
      rinv[j] = pow2i(-L);
      if (src[j] <= -2) {
        tm = L > tm ? L : tm;
        tn = L < tn ? L : tn;
      }
    }
  }
  if (tmax) {
    tm = __reduce_max_sync(0xffffffffu, tm);
    tn = __reduce_min_sync(0xffffffffu, tn);
    if ((wtid & 31) == 0 && tm != kNoExp) {
      atomicMax(tmax, tm);
      atomicMin(tmin, tn);
    }
  }
}

// Dequantise chunk c of a tile in place: every worker first reads the raw
// bytes of its items (8-dim groups, see chunk_item), then writes them as f16
// into the two 64-dim swizzle atoms of the chunk. Between the phases stands a
// barrier of the workers, or only of the warp where a chunk holds 128 code
// dims: there row j's raw bytes are [128 j, 128 j + 128), read by the 16
// items of row j (16 consecutive workers, one warp), and the only raw bytes
// any f16 write covers are those of its own row. `s2` holds each row's code
// multiplier and `rinv` its reciprocal row multiplier (see the top of the
// file and scale_multipliers). Rows without a source read stale bytes, which
// are discarded: they become zeros. Each warp's items are all codes or all
// bf16 (the layouts of the 448 + 64 entry and of window tokens), so the items
// of a thread run without per-item branches; other layouts take the general
// path.
DSV4_DEV void convert_chunk(const AttnArgs& a, bool win, const int32_t* src, const uint32_t* s2, const float* rinv,
                            int c, int rc, unsigned char* xc, int wtid, float& mx) {
  const ChunkSplit cs = chunk_split(a, c);
  const int nn = win ? 128 : cs.nn;   // window rows: the item layout of a full chunk
  const int n_items = rc * 16;
  const int warp_q = wtid >> 5;       // items of a thread share the parity of i >> 5 (kWorkers is a multiple of 64)
  const bool all_codes = !win && (cs.nn == 128 || (cs.nn == 64 && (warp_q & 1) == 0));
  const bool all_bf16 = win || cs.nn == 0 || (cs.nn == 64 && (warp_q & 1) == 1);
  uint4 rw[kItems];
  if (all_codes) {
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int i = wtid + it * kWorkers;
      int j, g;
      chunk_item(nn, i, j, g);
      rw[it] = make_uint4(0u, 0u, 0u, 0u);
      if (i < n_items) {
        const uint2 w = *reinterpret_cast<const uint2*>(xc + j * cs.nn + 8 * g);
        rw[it].x = w.x;
        rw[it].y = w.y;
      }
    }
  } else if (all_bf16) {
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int i = wtid + it * kWorkers;
      int j, g;
      chunk_item(nn, i, j, g);
      rw[it] = make_uint4(0u, 0u, 0u, 0u);
      if (i < n_items)
        rw[it] = *reinterpret_cast<const uint4*>(win ? xc + j * 256 + 16 * g
                                                      : xc + cs.rope_off + j * cs.rb + 2 * (8 * g - cs.nn));
    }
  } else {
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int i = wtid + it * kWorkers;
      int j, g;
      chunk_item(nn, i, j, g);
      rw[it] = make_uint4(0u, 0u, 0u, 0u);
      if (i < n_items && src[j] >= 0) {
        if (8 * g < cs.nn) {
          const uint2 w = *reinterpret_cast<const uint2*>(xc + j * cs.nn + 8 * g);
          rw[it].x = w.x;
          rw[it].y = w.y;
        } else {
          rw[it] = *reinterpret_cast<const uint4*>(xc + cs.rope_off + j * cs.rb + 2 * (8 * g - cs.nn));
        }
      }
    }
  }
  if (!win && cs.nn == 128) __syncwarp();
  else tc::bar_named(kBarWork, kWorkers);
  if (all_codes) {
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int i = wtid + it * kWorkers;
      int j, g;
      chunk_item(nn, i, j, g);
      if (i < n_items) {
        const bool valid = src[j] >= 0;
        const uint4 h = codes8_to_f16x8(make_uint2(rw[it].x, rw[it].y), s2[j]);
        store_group(xc, j, g, valid ? h : make_uint4(0u, 0u, 0u, 0u));
      }
    }
  } else if (all_bf16) {
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int i = wtid + it * kWorkers;
      int j, g;
      chunk_item(nn, i, j, g);
      if (i < n_items) {
        const int32_t sr = src[j];
        const bool valid = win ? sr <= -2 : sr >= 0;
        float m = 0.f;
        const uint4 h = bf16x8_to_f16x8_scaled(rw[it], rinv[j], m);
        mx = valid ? fmaxf(mx, m) : mx;
        store_group(xc, j, g, valid ? h : make_uint4(0u, 0u, 0u, 0u));
      }
    }
  } else {
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int i = wtid + it * kWorkers;
      if (i < n_items) {
        int j, g;
        chunk_item(nn, i, j, g);
        uint4 h = make_uint4(0u, 0u, 0u, 0u);
        if (src[j] >= 0) {
          if (8 * g < cs.nn) h = codes8_to_f16x8(make_uint2(rw[it].x, rw[it].y), s2[j]);
          else h = bf16x8_to_f16x8_scaled(rw[it], rinv[j], mx);
        }
        store_group(xc, j, g, h);
      }
    }
  }
}

// One producer thread: the TMA boxes of chunk c of compressed tile tl
// (contiguous rows) into the chunk's region, completing on xland[c].
DSV4_DEV void issue_tma_chunk(const AttnArgs& a, const AttnMaps& maps, int b, const Tile& tl, int c,
                              unsigned char* xk, uint64_t* xland, uint32_t* sk) {
  const int y = static_cast<int>(static_cast<int64_t>(b / a.T) * a.capacity + tl.r0);
  const ChunkSplit cs = chunk_split(a, c);
  unsigned char* xc = xk + c * kChunkBytes;
  // with the first chunk, the tile's scales (raw fp32, a whole number of
  // 16-byte granules: the capacity is a multiple of 4 on this path, so the
  // copy starts aligned and ends inside the sequence's rows)
  const uint32_t sbytes = c == 0 && sk ? static_cast<uint32_t>((tl.cnt + 3) & ~3) * 4u : 0u;
  tc::mbar_arrive_expect_tx(&xland[c], static_cast<uint32_t>(a.tile_rows * (cs.nn + cs.rb)) + sbytes);
  if (sbytes) tc::bulk_load(sk, a.k_scale + y, sbytes, &xland[c]);
  if (cs.nn == 128) tc::tma_load_2d(xc, &maps.nope, &xland[c], c * 128, y);
  else if (cs.nn > 0) tc::tma_load_2d(xc, &maps.nope_tail, &xland[c], c * 128, y);
  if (cs.rb > 0) tc::tma_load_2d(xc + cs.rope_off, &maps.rope, &xland[c], 0, y);
}

// In-warp reduce-scatter of 32 values per lane (one per head): afterwards v[0]
// holds the max (or sum) over the warp's 32 lanes for head `lane`. Each step
// keeps half of the values and takes the other half from the partner lane.
template <bool MAX>
DSV4_DEV void warp_reduce_scatter32(float* v, int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int half = 16 >> step;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

// Two in-warp reduce-scatter sums at once (independent shuffle chains):
// afterwards a[0] and b[0] hold the sums over the warp's 32 lanes for head
// `lane` of each array.
DSV4_DEV void warp_reduce_scatter32_sum2(float* a, float* b, int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int half = 16 >> step;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float sa = up ? a[i] : a[i + half], ka = up ? a[i + half] : a[i];
      const float sb = up ? b[i] : b[i + half], kb = up ? b[i + half] : b[i];
      const float ra = __shfl_xor_sync(0xffffffffu, sa, o);
      const float rb = __shfl_xor_sync(0xffffffffu, sb, o);
      a[i] = ka + ra;
      b[i] = kb + rb;
    }
  }
}

// 32 scores (heads [col, col + 32)) of this thread's row, scaled to the log2
// domain; -inf for a row that does not exist.
DSV4_DEV void load_scores32(uint32_t taddr, float c2, bool valid, float* s) {
  uint32_t v[32];
  tc::tmem_ld32(taddr, v);
  tc::tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) s[i] = valid ? __uint_as_float(v[i]) * c2 : -INFINITY;
}

// The query rows a worker loaded (8-dim bf16 groups, item i = wtid + u *
// workers, head i / gpr by the exact reciprocal qrcp) as f16 into the K-major
// operand qs; a value beyond f16 raises RANGE.
DSV4_DEV void stage_query(unsigned char* qs, const uint4* qw, int wtid, int gpr, uint32_t qrcp, int* status) {
  float qmax = 0.f;
#pragma unroll
  for (int u = 0; u < kQItems; ++u) {
    const int i = wtid + u * kWorkers;
    if (i < kHeads * gpr) {
      const int h = static_cast<int>(((static_cast<uint32_t>(i) >> 4) * qrcp) >> 16), d0 = (i - h * gpr) * 8;
      const int atom = d0 >> 6, gg = (d0 >> 3) & 7;
      *reinterpret_cast<uint4*>(qs + atom * kQAtomBytes + h * 128 + ((gg ^ (h & 7)) << 4)) =
          bf16x8_to_f16x8(qw[u], qmax);
    }
  }
  if (qmax >= kF16Max) atomicOr(status, DSV4_STATUS_RANGE);
}

}  // namespace

// grid (splits, B, head groups), block 512. See the top of the file.
template <bool SEP>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnMaps maps, AttnArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int D = a.D;
  const int nch = D / 128;
  unsigned char* qs = base;                                  // D/64 atoms of [64 heads][128 B]
  unsigned char* pb = qs + D * 128;                          // [128 rows][64 heads] f16
  unsigned char* xk = pb + kPBytes;                          // nch chunks of [2 atoms][128 rows][128 B]
  unsigned char* xv = SEP ? xk + nch * kChunkBytes : xk;
  TcTail* t = reinterpret_cast<TcTail*>(xk + (SEP ? 2 : 1) * nch * kChunkBytes);
  pdl_trigger();
  if (threadIdx.x == 32 && a.tma) {
    tc::prefetch_tensormap(&maps.nope);
    tc::prefetch_tensormap(&maps.nope_tail);
    tc::prefetch_tensormap(&maps.rope);
  }
  const int split = blockIdx.x, b = blockIdx.y;
  const int h0 = blockIdx.z * kHeads;
  const int hcount = a.H - h0 < kHeads ? a.H - h0 : kHeads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // workers: the query rows of this head group (bf16), all loads in flight
  // while the CTA waits for the previous kernel and sets up; converted into
  // the MMA operand further down. The query is an input no kernel of this
  // library writes, complete before the call's kernels start, so it is read
  // before the programmatic-launch wait.
  const int gpr = D / 8;   // 8-dim groups per head
  // head of query group i: i / gpr = (i / 16) / (D / 128) by an exact
  // reciprocal (exact for every i < 128 * gpr and D / 128 <= 16)
  const uint32_t qrcp = (65536u + (D >> 7) - 1) / static_cast<uint32_t>(D >> 7);
  uint4 qw[kQItems];
  if (warp >= 2) {
    const int wtid = threadIdx.x - 64;
#pragma unroll
    for (int u = 0; u < kQItems; ++u) {
      const int i = wtid + u * kWorkers;
      const int h = static_cast<int>(((static_cast<uint32_t>(i) >> 4) * qrcp) >> 16);
      qw[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i < kHeads * gpr && h < hcount)
        qw[u] = __ldg(reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(b) * a.H + h0 + h) * D) +
                      (i - h * gpr));
    }
  }
  // CSA CTAs start long before the top-k they read is done: they stage the
  // query in the meantime (HCA CTAs start just before the append ends, and
  // stage it after the setup).
  const bool q_early = a.n_sel != 0;
  if (q_early && warp >= 2) stage_query(qs, qw, threadIdx.x - 64, gpr, qrcp, a.status);
  pdl_wait();

  const RowSpace rs = row_space(a, b);
  const int tile0 = split * a.tiles_per_split;
  const int tiles = rs.mt + rs.wt;
  const int nt = tiles - tile0 < a.tiles_per_split ? (tiles - tile0 > 0 ? tiles - tile0 : 0) : a.tiles_per_split;
  if (nt == 0) {   // uniform: nothing to attend in this split
    for (int h = threadIdx.x; h < hcount; h += blockDim.x) {
      a.part_lse[(static_cast<int64_t>(b) * a.H + h0 + h) * a.splits + split] = -INFINITY;
      a.part_lsev[(static_cast<int64_t>(b) * a.H + h0 + h) * a.splits + split] = -INFINITY;
    }
    return;
  }

  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(kHeads * (1 + nch))) cols <<= 1;
  volatile int* abort = &t->abort;

  if (warp == 0) tc::tmem_alloc(&t->taddr, cols);
  const Tile first = tile_at(a, rs, tile0);
  const bool first_tma = !SEP && a.tma && !first.win;
  if (threadIdx.x == 32) {
    for (int c = 0; c < kMaxChunks; ++c) {
      tc::mbar_init(&t->xland[c], 1);
      tc::mbar_init(&t->xfull[c], kWorkers / 32);
      tc::mbar_init(&t->xfree[c], 1);
    }
    tc::mbar_init(&t->sfull, 1);
    tc::mbar_init(&t->pfull, kSoftThreads / 32);
    tc::mbar_init(&t->qready, kWorkers / 32);
    tc::mbar_init(&t->drain, 1);
    tc::mbar_init(&t->never, 1);
    t->abort = 0;
    tc::fence_mbar_init();
  }
  if (threadIdx.x < kHeads) {
    t->m_used[threadIdx.x] = -INFINITY;
    t->mv_used[threadIdx.x] = -INFINITY;
  }
  if (threadIdx.x < kMaxTiles) {
    t->texv[threadIdx.x] = kNoExp;
    t->texn[threadIdx.x] = -kNoExp;
  }
  float* const rmul = row_muls<SEP>(t);
  // Row sources of every tile of the split (CSA: one round trip for the top-k
  // indices). Each tile's scales travel with its first chunk: a bulk copy
  // beside the TMA boxes (contiguous rows, capacity a multiple of 4) or one
  // 4-byte copy per gathered row; otherwise they are loaded here.
  const bool bulk_scales = !SEP && a.tma && (a.capacity & 3) == 0;
  int32_t sr[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = threadIdx.x + k * kThreads, tt = i >> 7;
    sr[k] = tt < nt ? row_source(a, rs, b, tile_at(a, rs, tile0 + tt), i & (kRows - 1)) : -1;
    if (tt < nt) t->src[i] = sr[k];
  }
  if (!SEP && a.tma && !bulk_scales) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = threadIdx.x + k * kThreads, tt = i >> 7;
      if (tt < nt && !tile_at(a, rs, tile0 + tt).win) t->sk[i] = __float_as_uint(sr[k] >= 0 ? __ldg(a.k_scale + sr[k]) : 0.f);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (first_tma && threadIdx.x == 32)
    for (int c = 0; c < nch; ++c)
      issue_tma_chunk(a, maps, b, first, c, xk, t->xland, bulk_scales ? t->sk : nullptr);
  if (!first_tma && warp >= 2) {
    const int wtid = threadIdx.x - 64;
    const int rc = (first.cnt + 15) & ~15;
    for (int c = 0; c < nch; ++c) {
      issue_chunk(a, b, first.win, t->src, c, rc, a.k_nope, a.k_rope, a.k_scale, a.win_k, xk + c * kChunkBytes, t->sk, wtid);
      if (SEP)
        issue_chunk(a, b, first.win, t->src, c, rc, a.v_nope, a.v_rope, a.v_scale, a.win_v, xv + c * kChunkBytes, t->sv, wtid);
      cp_async_commit();
    }
  }
  const uint32_t taddr = t->taddr;
  const uint32_t s_tmem = taddr, o_tmem = taddr + kHeads;
  const int32_t* src = t->src;

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_f16_f32(kRows, kHeads, 0, 0);
      const uint32_t id_pv = tc::idesc_f16_f32(kRows, kHeads, 1, 1);
      const uint32_t q_sa = tc::smem_u32(qs), p_sa = tc::smem_u32(pb);
      const uint32_t xk_sa = tc::smem_u32(xk), xv_sa = tc::smem_u32(xv);
      bool ok = true;
      if (g_force_timeout) ok = tc::mbar_wait_for(&t->never, 0, abort, kForcedWaitNs);   // test hook: runs out
      ok = ok && tc::mbar_wait(&t->qready, 0, abort);
      for (int tt = 0; ok && tt < nt; ++tt) {
        const int kk_pv = (tile_at(a, rs, tile0 + tt).cnt + 15) >> 4;   // 16-row steps holding rows
        for (int c = 0; c < nch; ++c) {
          if (!(ok = tc::mbar_wait(&t->xfull[c], tt & 1, abort))) break;
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
            const uint64_t ad = tc::smem_desc(xk_sa + c * kChunkBytes + koff, 1024, tc::kSwizzle128B);
            const uint64_t bd =
                tc::smem_desc(q_sa + (2 * c + (kk >> 2)) * kQAtomBytes + (kk & 3) * 32, 1024, tc::kSwizzle128B);
            tc::mma_f16(s_tmem, ad, bd, id_qk, (c | kk) ? 1u : 0u);
          }
        }
        if (!ok) break;
        tc::tc_commit(&t->sfull);
        if (!(ok = tc::mbar_wait(&t->pfull, tt & 1, abort))) break;
        tc::tc_fence_after();
        for (int c = 0; c < nch; ++c) {
          for (int kk = 0; kk < kk_pv; ++kk) {
            const uint64_t ad =
                tc::smem_desc_lbo(xv_sa + c * kChunkBytes + kk * 2048, kAtomBytes, 1024, tc::kSwizzle128B);
            const uint64_t bd = tc::smem_desc_lbo(p_sa + kk * 2048, kAtomBytes, 1024, tc::kSwizzle128B);
            tc::mma_f16(o_tmem + c * kHeads, ad, bd, id_pv, (tt | kk) ? 1u : 0u);
          }
          tc::tc_commit(&t->xfree[c]);
        }
      }
      // every MMA issued must finish before tensor memory is released
      tc::tc_commit(&t->drain);
      tc::mbar_wait_drain(&t->drain, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ TMA producer (HCA compressed rows)
    if (!SEP && a.tma) {
      const int64_t row_base = static_cast<int64_t>(b / a.T) * a.capacity;
      if (lane == 0) {
        // boxes issued per chunk (the first tile's went out before the setup)
        int issued[kMaxChunks];
        for (int c = 0; c < kMaxChunks; ++c) issued[c] = first_tma ? 1 : 0;
        bool ok = true;
        for (int tt = first_tma ? 1 : 0; ok && tt < nt; ++tt) {
          const Tile tl = tile_at(a, rs, tile0 + tt);
          if (tl.win) break;   // window tiles come last and go by cp.async
          for (int c = 0; c < nch; ++c) {
            if (!(ok = tc::mbar_wait(&t->xfree[c], (tt - 1) & 1, abort))) break;
            issue_tma_chunk(a, maps, b, tl, c, xk, t->xland, bulk_scales ? t->sk + tt * kRows : nullptr);
            ++issued[c];
          }
        }
        // every box issued must land before the CTA's shared memory goes away
        for (int c = 0; c < nch; ++c)
          if (issued[c] > 0) tc::mbar_wait_drain(&t->xland[c], (issued[c] - 1) & 1);
      } else if (nt > 1 && (lane == 1 || lane == 2)) {
        // later tiles' compressed rows into L2 (the first tile's boxes are on
        // their way); after the query has arrived, so that it is not queued
        // behind them
        const Tile t1 = tile_at(a, rs, tile0 + 1);
        const Tile tl = tile_at(a, rs, tile0 + nt - 1);
        if (!t1.win && tc::mbar_wait(&t->qready, 0, abort)) {
          const int64_t e0 = row_base + t1.r0;
          const int64_t n = (tl.win ? rs.n_main : tl.r0 + tl.cnt) - t1.r0;
          if (lane == 1) tc::prefetch_l2_range(a.k_nope + e0 * a.d_nope, n * a.d_nope);
          if (lane == 2 && a.d_rope) tc::prefetch_l2_range(a.k_rope + e0 * a.d_rope, n * a.d_rope * 2);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ workers (warps 2-15)
    const int wtid = threadIdx.x - 64;
    const bool soft = (warp >= 4 && warp < 8) || warp >= 12;
    const int qd = warp & 3;                       // tensor-memory lane quarter
    const int hb = warp >= 12 ? 32 : 0;            // a softmax warp's heads [hb, hb + 32)
    const int j = qd * 32 + lane;                  // row of the tile / dim of an O^T block
    const int st = (warp >= 12 ? 128 : 0) + qd * 32 + lane;   // 0..255 among the softmax threads
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const float c2 = a.sm_scale * 1.4426950408889634f;
    float mx = 0.f;

    {
      // the query, bf16 -> f16 into the K-major operand (heads beyond H zero)
      if (!q_early) stage_query(qs, qw, wtid, gpr, qrcp, a.status);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&t->qready);
    }

    float lw = 0.f;   // softmax warps: l of head hb + lane over this warp's rows
    float lv = 0.f;   // and l' (the sum of the value-side weights P)
    // Every worker takes part in the same sequence of worker barriers; a
    // softmax failure (a wait that gave up) reaches the others through the
    // next one, so no worker is left waiting at a named barrier.
    bool ok = true, soft_ok = true;
    for (int tt = 0; ok && tt < nt; ++tt) {
      const Tile tl = tile_at(a, rs, tile0 + tt);
      const int rc = (tl.cnt + 15) & ~15;
      const bool via_tma = !SEP && a.tma && !tl.win;
      const int32_t* src_t = src + tt * kRows;
      if (!via_tma && tt > 0) {
        for (int c = 0; c < nch; ++c) {
          const bool w = soft_ok && tc::mbar_wait(&t->xfree[c], (tt - 1) & 1, abort);
          if (!(ok = tc::bar_and(kBarWork, kWorkers, w))) break;
          issue_chunk(a, b, tl.win, src_t, c, rc, a.k_nope, a.k_rope, a.k_scale, a.win_k, xk + c * kChunkBytes,
                      t->sk + tt * kRows, wtid);
          if (SEP)
            issue_chunk(a, b, tl.win, src_t, c, rc, a.v_nope, a.v_rope, a.v_scale, a.win_v, xv + c * kChunkBytes,
                        t->sv + tt * kRows, wtid);
          cp_async_commit();
        }
        if (!ok) break;
      }
      float* const rik = rmul + tt * kRows;                        // 1 / mu of the key (or shared) rows
      float* const riv = SEP ? rik + kMulsPerSplit : rik;          // of the value rows
      for (int c = 0; c < nch; ++c) {
        bool w = soft_ok;
        if (via_tma) w = w && tc::mbar_wait(&t->xland[c], tt & 1, abort);
        else cp_async_wait(tl.win ? 0 : nch - 1 - c);
        // The rows' exponents. Every worker takes part whatever its w (the
        // warp-wide reductions need whole warps; data read after a failed wait
        // is garbage that the failed barrier below discards). A compressed
        // tile's scales came with its first chunk (each row's by the worker that
        // reads it here); a window tile needs whole rows: every worker waited
        // for all its copies of the tile above, and after this barrier
        // everyone's have landed, read before any chunk converts.
        if (c == 0 && !tl.win) {
          scale_multipliers(src_t, t->sk + tt * kRows, rc, wtid, rik, SEP ? nullptr : &t->texv[tt], &t->texn[tt]);
          if (SEP) scale_multipliers(src_t, t->sv + tt * kRows, rc, wtid, riv, &t->texv[tt], &t->texn[tt]);
        }
        if (c == 0 && tl.win) {
          tc::bar_named(kBarWork, kWorkers);
          window_multipliers(xk, src_t, nch, rc, wtid, rik, SEP ? nullptr : &t->texv[tt], &t->texn[tt]);
          if (SEP) window_multipliers(xv, src_t, nch, rc, wtid, riv, &t->texv[tt], &t->texn[tt]);
        }
        // every worker's copies of chunk c have landed (or the boxes have)
        if (!(ok = tc::bar_and(kBarWork, kWorkers, w))) break;
        convert_chunk(a, tl.win, src_t, t->sk + tt * kRows, rik, c, rc, xk + c * kChunkBytes, wtid, mx);
        if (SEP) {
          tc::bar_named(kBarWork, kWorkers);
          convert_chunk(a, tl.win, src_t, t->sv + tt * kRows, riv, c, rc, xv + c * kChunkBytes, wtid, mx);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&t->xfull[c]);
      }
      if (!ok || !soft) continue;

      // ---- softmax warps: S^T -> P for this tile
      const bool valid = src_t[j] != -1;
      const float mkj = __frcp_rn(rik[j]);          // the key row's multiplier mu_j
      const float ck = c2 * mkj;                    // ... back on its scores
      const float mvj = SEP ? __frcp_rn(riv[j]) : mkj;   // the value row's multiplier mu'_j
      const float fv = static_cast<float>(binade(mvj));          // L'_j
      const int tv = t->texv[tt] == kNoExp ? 0 : t->texv[tt];   // T, the tile's largest L'
      const float rj = valid ? mvj * pow2i(-tv) : 0.f;          // mu'_j / 2^T < 2
      float* const phi = t->phi[tt & 1];
      // The head's power of two 2^(T + m - M) for this tile (recomputed below
      // when a max moves). Tile tt - 2 used the same slot; every softmax thread
      // finished with it before the barrier of tile tt - 1, which this thread
      // has passed.
      if (st < kHeads) {
        const float mo = t->m_used[st], vo = t->mv_used[st];
        phi[st] = (mo == -INFINITY || vo == -INFINITY) ? 0.f : pow2_clamped(tv + static_cast<int>(mo - vo));
      }
      if (!(soft_ok = tc::bar_and(kBarSoft, kSoftThreads, tc::mbar_wait(&t->sfull, tt & 1, abort)))) continue;
      tc::tc_fence_after();
      float s[32];
      load_scores32(s_tmem + lane_off + hb, ck, valid, s);
      // A max moves when s > m + 2^8 or s + L' > M + 2^8; on a CTA's first
      // tile they always do (both start at -inf).
      bool need = tt == 0;
      if (tt > 0) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 mu = *reinterpret_cast<const float4*>(t->m_used + hb + i);
          const float4 mv = *reinterpret_cast<const float4*>(t->mv_used + hb + i);
          need |= (s[i] > fminf(mu.x, mv.x - fv) + kRescale) | (s[i + 1] > fminf(mu.y, mv.y - fv) + kRescale) |
                  (s[i + 2] > fminf(mu.z, mv.z - fv) + kRescale) | (s[i + 3] > fminf(mu.w, mv.w - fv) + kRescale);
        }
      }
      if (tc::bar_or(kBarSoft, kSoftThreads, need)) {
        // a running max of some head moves: reduce this tile's column max of s,
        // and of s + L' unless the tile's L' lie within 2^8 of each other: then
        // max(s) + T bounds it closely enough (the largest P of the tile stays
        // >= 2^-9); the maxima kept are integers, so every rescale is an exact
        // power of two
        const bool exact_v = t->texv[tt] - t->texn[tt] > static_cast<int>(kRescale);
        float v[32];
        if (exact_v) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = s[i] + fv;
          warp_reduce_scatter32<true>(v, lane);
          t->redv[qd][hb + lane] = v[0];
        }
        warp_reduce_scatter32<true>(s, lane);
        t->red[qd][hb + lane] = s[0];
        tc::bar_named(kBarSoft, kSoftThreads);
        if (st < kHeads) {
          const float tm = fmaxf(fmaxf(t->red[0][st], t->red[1][st]), fmaxf(t->red[2][st], t->red[3][st]));
          const float tvm = exact_v ? fmaxf(fmaxf(t->redv[0][st], t->redv[1][st]), fmaxf(t->redv[2][st], t->redv[3][st]))
                                    : tm + static_cast<float>(tv);
          const float mo = t->m_used[st], mn = fmaxf(mo, ceilf(tm));
          const float vo = t->mv_used[st], vn = fmaxf(vo, ceilf(tvm));
          t->alpha[st] = pow2_diff(mo, mn);
          t->alphav[st] = pow2_diff(vo, vn);
          t->m_used[st] = mn;
          t->mv_used[st] = vn;
          phi[st] = (mn == -INFINITY || vn == -INFINITY) ? 0.f : pow2_clamped(tv + static_cast<int>(mn - vn));
        }
        tc::bar_named(kBarSoft, kSoftThreads);
        lw *= t->alpha[hb + lane];
        lv *= t->alphav[hb + lane];
        if (tt > 0) {
          for (int c = 0; c < nch; ++c) {
            uint32_t o[32];
            const uint32_t addr = o_tmem + lane_off + c * kHeads + hb;
            tc::tmem_ld32(addr, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * t->alphav[hb + i]);
            tc::tmem_st32(addr, o);
          }
          tc::tmem_wait_st();
        }
        load_scores32(s_tmem + lane_off + hb, ck, valid, s);   // the reduction consumed s
      }
      // p = 2^(s - m) (for l) and the value-side weight P = p * mu' / 2^T *
      // 2^(T + m - M), as f16 into P (row j, 16-byte chunks, swizzled)
      float pr[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 mu = *reinterpret_cast<const float4*>(t->m_used + hb + i);
        s[i] = valid ? ex2(s[i] - mu.x) : 0.f;
        s[i + 1] = valid ? ex2(s[i + 1] - mu.y) : 0.f;
        s[i + 2] = valid ? ex2(s[i + 2] - mu.z) : 0.f;
        s[i + 3] = valid ? ex2(s[i + 3] - mu.w) : 0.f;
        pr[i] = s[i] * rj;
        pr[i + 1] = s[i + 1] * rj;
        pr[i + 2] = s[i + 2] * rj;
        pr[i + 3] = s[i + 3] * rj;
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int i = g * 8, gc = (hb >> 3) + g;
        const float4 fa = *reinterpret_cast<const float4*>(phi + hb + i);
        const float4 fb = *reinterpret_cast<const float4*>(phi + hb + i + 4);
        *reinterpret_cast<uint4*>(pb + j * 128 + ((gc ^ (j & 7)) << 4)) = make_uint4(
            f32x2_to_f16x2(pr[i] * fa.x, pr[i + 1] * fa.y), f32x2_to_f16x2(pr[i + 2] * fa.z, pr[i + 3] * fa.w),
            f32x2_to_f16x2(pr[i + 4] * fb.x, pr[i + 5] * fb.y), f32x2_to_f16x2(pr[i + 6] * fb.z, pr[i + 7] * fb.w));
      }
      warp_reduce_scatter32_sum2(s, pr, lane);
      lw += s[0];
      lv += pr[0] * phi[hb + lane];   // l' of head hb + lane
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&t->pfull);
    }
    cp_async_wait(0);
    if (mx >= kF16Max) atomicOr(a.status, DSV4_STATUS_RANGE);

    if (soft) {
      // ---- epilogue: normalise O^T and store this split's f16 partial [D][64 heads]
      ok = tc::bar_and(kBarSoft, kSoftThreads, ok && soft_ok);
      if (ok) {
        t->red[qd][hb + lane] = lw;
        t->redv[qd][hb + lane] = lv;
        tc::bar_named(kBarSoft, kSoftThreads);
        if (st < kHeads) {
          const float l = (t->red[0][st] + t->red[1][st]) + (t->red[2][st] + t->red[3][st]);
          const float lvs = (t->redv[0][st] + t->redv[1][st]) + (t->redv[2][st] + t->redv[3][st]);
          t->lsum[st] = l;
          t->lvsum[st] = lvs;
          t->alpha[st] = lvs > 0.f ? 1.f / lvs : 0.f;
        }
        tc::bar_named(kBarSoft, kSoftThreads);
        if (st < hcount) {
          const float l = t->lsum[st], lvs = t->lvsum[st];
          const int64_t o = (static_cast<int64_t>(b) * a.H + h0 + st) * a.splits + split;
          a.part_lse[o] = l > 0.f ? (t->m_used[st] + __log2f(l)) * 0.6931471805599453f : -INFINITY;
          a.part_lsev[o] = lvs > 0.f && l > 0.f ? (t->mv_used[st] + __log2f(lvs)) * 0.6931471805599453f : -INFINITY;
        }
        // O^T / l' as f16 rows [dim][64 heads], 16-byte granule q of row r
        // at granule q ^ (r & 7) (the merge reads the same swizzle), stored
        // straight from registers: each thread writes 64 contiguous bytes of
        // its dim's row. A 128-dim block is stored as soon as the last tile's
        // P.V of that block has finished, overlapping the remaining MMAs.
        const int hgs = gridDim.z;
        unsigned char* part = reinterpret_cast<unsigned char*>(a.part_o) +
                              ((static_cast<int64_t>(b) * a.splits + split) * hgs + blockIdx.z) * D * kHeads * 2;
        for (int c = 0; ok && c < nch; ++c) {
          if (!(ok = tc::bar_and(kBarSoft, kSoftThreads, tc::mbar_wait(&t->xfree[c], (nt - 1) & 1, abort)))) break;
          tc::tc_fence_after();
          uint32_t v[32];
          tc::tmem_ld32(o_tmem + lane_off + c * kHeads + hb, v);
          tc::tmem_wait_ld();
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float4 al = *reinterpret_cast<const float4*>(t->alpha + hb + 2 * i);
            w[i] = f32x2_to_f16x2(__uint_as_float(v[2 * i]) * al.x, __uint_as_float(v[2 * i + 1]) * al.y);
            w[i + 1] = f32x2_to_f16x2(__uint_as_float(v[2 * i + 2]) * al.z, __uint_as_float(v[2 * i + 3]) * al.w);
          }
          const int r = c * 128 + j;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            *reinterpret_cast<uint4*>(part + r * 128 + ((((hb >> 3) + q4) ^ (r & 7)) << 4)) =
                make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
        }
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(taddr, cols);
  }
  if (threadIdx.x == 0 && t->abort) atomicOr(a.status, DSV4_STATUS_TIMEOUT);
}

namespace {

size_t tc_smem_bytes(int D, bool sep) {
  return 1024 + static_cast<size_t>(D) * 128 + kPBytes + (sep ? 2 : 1) * static_cast<size_t>(D / 128) * kChunkBytes +
         sizeof(TcTail) + (sep ? 2 * kMulsPerSplit * sizeof(float) : 0);
}

template <bool SEP>
int launch_tc(const AttnMaps& maps, const AttnArgs& a, int head_groups, cudaStream_t st) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(attn_tc_kernel<SEP>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  const size_t smem = tc_smem_bytes(a.D, SEP);
  return launch_pdl(attn_tc_kernel<SEP>, dim3(a.splits, a.B, head_groups), dim3(kThreads), smem, st, maps, a);
}

}  // namespace

int attention_force_timeout(int on) {
  const int v = on ? 1 : 0;
  return cudaMemcpyToSymbol(g_force_timeout, &v, sizeof(v)) == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

bool attention_tc_supported(int H, int d_nope, int d_rope, int separate_v) {
  const int D = d_nope + d_rope;
  if (H < 1 || H > 128 || D % 128 || D > 128 * kMaxChunks || d_nope % 16 || d_rope % 8) return false;
  if (separate_v && D > 256) return false;
  return tc_smem_bytes(D, separate_v != 0) <= 227 * 1024;
}

bool attention_tc_tma_shape(int d_nope, int d_rope, int separate_v) {
  // every chunk but the last holds 128 codes; the last holds the remaining
  // codes and all RoPE dims (so three box shapes cover every load)
  return !separate_v && d_rope <= 128 && (d_rope == 0 || d_nope % 128 + d_rope == 128);
}

int launch_attention_tc(const AttnArgs& a0, int head_groups, cudaStream_t st) {
  AttnArgs a = a0;
  AttnMaps maps;
  memset(&maps, 0, sizeof(maps));
  a.tma = 0;
  if (a.n_sel == 0 && attention_tc_tma_shape(a.d_nope, a.d_rope, a.separate_v)) {
    const int64_t rows = static_cast<int64_t>(a.B / a.T) * a.capacity;
    const int tail = a.d_nope % 128;
    bool ok = a.d_nope < 128 || encode_u8_rows(&maps.nope, a.k_nope, rows, a.d_nope, 128, a.tile_rows);
    if (ok && tail) ok = encode_u8_rows(&maps.nope_tail, a.k_nope, rows, a.d_nope, tail, a.tile_rows);
    if (ok && a.d_rope) ok = encode_u8_rows(&maps.rope, a.k_rope, rows, 2 * a.d_rope, 2 * a.d_rope, a.tile_rows);
    a.tma = ok ? 1 : 0;
  }
  const int e = a.separate_v ? launch_tc<true>(maps, a, head_groups, st) : launch_tc<false>(maps, a, head_groups, st);
  if (e) return e;
  return launch_attention_merge_tc(a, head_groups, st);
}

}  // namespace dsv4
