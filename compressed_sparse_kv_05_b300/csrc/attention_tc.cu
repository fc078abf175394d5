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
// contractions per tile of 128 rows:
//   X   [128 rows][D]  f16: each row's dequantised key (code * scale || rope, or
//                      the raw window token); it is also the value row when K = V
//   S^T [128][64]      = X . Q^T             (M = 128 rows, N = 64 heads, K = D)
//   P   [128][64]      = exp2(S^T * c - m)   (f16, the running max m per head)
//   O^T [D][64]       += X^T . P             (M = 128 dims per block, N = 64, K = 128 rows)
// X is written once per tile in the 128-byte-swizzled layout that serves as a
// K-major operand for the first product and as an MN-major operand for the
// second; S^T and O^T live in tensor memory (lane = row / dim, column = head).
//
// CTA roles (512 threads, one CTA per SM for D = 512):
//   warp 0      allocates tensor memory, prefetches the CTA's rows into L2, and
//               one lane issues every MMA;
//   warps 1-3, 8-11   (224 threads) dequantise rows into X, chunk by chunk of
//               128 dims, with the loads of the next chunk in flight. An e4m3
//               code becomes f16 by integer operations (its bit pattern shifted
//               into an f16 is exactly code * 2^-8) and one f16 multiply by the
//               row's scale * 2^8;
//   warps 4-7, 12-15  (two per 32-lane quarter of tensor memory: one row each,
//               heads 0-31 or 32-63) convert the query, then turn S^T into P.
//               The running max of a head only moves when a score exceeds it by
//               more than 2^8 (then the tile's column max is reduced and O^T
//               and l are rescaled), so P <= 256 always fits f16. After the
//               last tile they normalise O^T, stage it in shared memory and
//               store this split's partial output with bulk copies.
// Splits are merged by attn_merge_kernel (attention.cu).
//
// Precision: K, V and P are rounded to f16 (relative error <= 2^-11 each; a
// row's scale is rounded to f16 once), the bf16 query converts to f16 exactly
// for |q| in [2^-14, 65504]; products and sums are fp32. A value that does not
// fit f16 (|x| >= 65504) raises DSV4_STATUS_RANGE. The two e4m3 NaN codes, which
// the quantiser never writes, read as +-480.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace dsv4 {

namespace {

constexpr int kRows = 128;                     // rows per tile
constexpr int kHeads = 64;                     // heads per CTA (MMA N), zero-padded
constexpr int kThreads = 512;
constexpr int kConvThreads = 7 * 32;           // warps 1-3 and 8-11
constexpr int kSoftThreads = 8 * 32;           // warps 4-7 and 12-15
constexpr int kGroups = kRows * 16;            // 8-dim groups of one 128-dim chunk
constexpr int kItems = (kGroups + kConvThreads - 1) / kConvThreads;
constexpr int kAtomBytes = kRows * 128;        // 128 rows x 64 dims f16
constexpr int kChunkBytes = 2 * kAtomBytes;    // 128 rows x 128 dims f16
constexpr int kQAtomBytes = kHeads * 128;      // 64 heads x 64 dims f16
constexpr int kPBytes = kRows * kHeads * 2;
constexpr int kMaxChunks = 4;                  // D <= 512
constexpr int kMaxTiles = 8;                   // rows per CTA <= 1024 (the host plan keeps to it)
constexpr int kBarSoft = 1, kBarConv = 2;      // named barriers (0 is __syncthreads)
constexpr float kRescale = 8.f;                // lazy-rescale threshold (log2 units)
constexpr float kF16Max = 65504.f;

struct TcTail {
  uint64_t xfull[kMaxChunks], xfree[kMaxChunks], sfull, pfull, pvdone, qready, qraw, drain;
  uint32_t taddr;
  int abort;
  int32_t src[kMaxTiles * kRows];   // row sources of every row of the split (see row_source)
  float sk[kMaxTiles * kRows];      // key (or shared entry) scale of every row, 0 for others
  float sv[kMaxTiles * kRows];      // value scale (separate V)
  float m_used[kHeads];             // running max per head, log2 domain
  float alpha[kHeads];
  float lsum[kHeads];
  float red[4][kHeads];
};

DSV4_DEV uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two e4m3 codes (bytes 0 and 1 of w after `sel`) as two f16 times f16x2 `sc`:
// placing code c in the low byte of a halfword, (c + (c & 0x80)) << 7 is the
// f16 bit pattern of e4m3(c) * 2^-8 (the sign moves to bit 15, the exponent and
// mantissa land under f16's, subnormals included).
DSV4_DEV uint32_t e4m3x2_to_f16x2_scaled(uint32_t w, uint32_t sel, uint32_t sc) {
  uint32_t h, r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(h) : "r"(w), "r"(sel));
  h = (h + (h & 0x00800080u)) << 7;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(sc));
  return r;
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

DSV4_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Rows of sequence b are numbered: first the compressed entries (the top-k list
// for CSA, every entry for HCA), then the window tokens, oldest first.
struct RowSpace {
  int64_t n_tok, n_c, n_win, n_main, R;
};

DSV4_DEV RowSpace row_space(const AttnArgs& a, int b) {
  RowSpace s;
  s.n_tok = a.n_tokens[b];
  s.n_c = s.n_tok / a.ratio < a.capacity ? s.n_tok / a.ratio : a.capacity;
  s.n_win = s.n_tok < a.window ? s.n_tok : a.window;
  s.n_main = a.n_sel > 0 ? a.n_sel : s.n_c;
  s.R = s.n_main + s.n_win;
  return s;
}

// Source of row r: >= 0 entry index into the planes (b * capacity + e), -1 no
// row (past the split, a -1 top-k slot or an invalid index), <= -2 window ring
// slot (-2 - slot).
DSV4_DEV int32_t row_source(const AttnArgs& a, const RowSpace& s, int b, int64_t r, int64_t r1, bool flag_bad) {
  if (r >= r1) return -1;
  if (r < s.n_main) {
    const int64_t e = a.n_sel > 0 ? static_cast<int64_t>(a.topk[static_cast<int64_t>(b) * a.n_sel + r]) : r;
    if (e < -1 || e >= s.n_c) {
      if (flag_bad) atomicOr(a.status, DSV4_STATUS_BAD_INDEX);
      return -1;
    }
    if (e < 0) return -1;
    return static_cast<int32_t>(static_cast<int64_t>(b) * a.capacity + e);
  }
  const int64_t pos = s.n_tok - s.n_win + (r - s.n_main);
  return static_cast<int32_t>(-2 - pos % a.window);
}

// [p, p + bytes) into L2, both ends rounded down to 16 bytes (never past the range).
DSV4_DEV void prefetch_range(const void* p, int64_t bytes) {
  const uintptr_t lo = (reinterpret_cast<uintptr_t>(p) + 15) & ~static_cast<uintptr_t>(15);
  const uintptr_t hi = (reinterpret_cast<uintptr_t>(p) + bytes) & ~static_cast<uintptr_t>(15);
  for (uintptr_t x = lo; x < hi; x += (1u << 20)) {
    const uintptr_t n = hi - x < (1u << 20) ? hi - x : (1u << 20);
    tc::prefetch_l2_bulk(reinterpret_cast<const void*>(x), static_cast<uint32_t>(n));
  }
}

// Warp 0: hint L2 to fetch every byte this CTA's rows [r0, r1) read.
DSV4_DEV void prefetch_rows(const AttnArgs& a, const RowSpace& s, int b, int64_t r0, int64_t r1, bool sep, int lane) {
  const int64_t m1 = r1 < s.n_main ? r1 : s.n_main;
  const int64_t base = static_cast<int64_t>(b) * a.capacity;
  if (m1 > r0) {
    if (a.n_sel == 0) {
      const int64_t e0 = base + r0, n = m1 - r0;
      if (lane == 0) prefetch_range(a.k_nope + e0 * a.d_nope, n * a.d_nope);
      if (lane == 1 && a.d_rope) prefetch_range(a.k_rope + e0 * a.d_rope, n * a.d_rope * 2);
      if (lane == 2) prefetch_range(a.k_scale + e0, n * 4);
      if (sep && lane == 3) prefetch_range(a.v_nope + e0 * a.d_nope, n * a.d_nope);
      if (sep && lane == 4 && a.d_rope) prefetch_range(a.v_rope + e0 * a.d_rope, n * a.d_rope * 2);
      if (sep && lane == 5) prefetch_range(a.v_scale + e0, n * 4);
    } else {
      for (int64_t r = r0 + lane; r < m1; r += 32) {
        const int64_t e = a.topk[static_cast<int64_t>(b) * a.n_sel + r];
        if (e < 0 || e >= s.n_c) continue;
        const int64_t row = base + e;
        prefetch_range(a.k_nope + row * a.d_nope, a.d_nope);
        if (a.d_rope) prefetch_range(a.k_rope + row * a.d_rope, a.d_rope * 2);
        if (sep) {
          prefetch_range(a.v_nope + row * a.d_nope, a.d_nope);
          if (a.d_rope) prefetch_range(a.v_rope + row * a.d_rope, a.d_rope * 2);
        }
      }
    }
  }
  const int64_t w0 = r0 > s.n_main ? r0 : s.n_main;
  if (r1 > w0 && lane < (sep ? 4 : 2)) {
    const int64_t pos0 = s.n_tok - s.n_win + (w0 - s.n_main);
    const int64_t cnt = r1 - w0, s0 = pos0 % a.window;
    const int64_t seg1 = cnt < a.window - s0 ? cnt : a.window - s0;
    const uint16_t* win = (lane >> 1) ? a.win_v : a.win_k;
    const int64_t rowb = static_cast<int64_t>(a.D) * 2;
    if ((lane & 1) == 0) prefetch_range(win + (static_cast<int64_t>(b) * a.window + s0) * a.D, seg1 * rowb);
    else if (cnt > seg1) prefetch_range(win + static_cast<int64_t>(b) * a.window * a.D, (cnt - seg1) * rowb);
  }
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

// Dims [128c, 128c + 128) of a row: nn FP8 dims (codes), the rest RoPE (bf16).
struct ChunkSplit {
  int nn, rope0;   // nope dims in the chunk; first RoPE dim (index into the row's RoPE part)
};
DSV4_DEV ChunkSplit chunk_split(const AttnArgs& a, int c) {
  const int n0 = c * 128;
  int nn = a.d_nope - n0;
  nn = nn < 0 ? 0 : (nn > 128 ? 128 : nn);
  return ChunkSplit{nn, n0 + nn - a.d_nope};
}

// Issue the asynchronous copies of chunk c of tile tt into the X chunk region
// `xc`: row j's raw bytes land at xc + 256 j, as the chunk's FP8 codes followed
// by its RoPE dims (bf16) for an entry, or its 128 bf16 values for a window
// token; rows that do not exist get nothing. Thread ctid copies 16-byte
// granules (row i / 16, granule i % 16) of its items.
DSV4_DEV void issue_chunk(const AttnArgs& a, int b, const int32_t* src, int tt, int c, const uint8_t* nope,
                          const uint16_t* rope, const uint16_t* win, unsigned char* xc, int ctid) {
  const ChunkSplit cs = chunk_split(a, c);
  const int ng = cs.nn / 16, ngr = (128 - cs.nn) / 8;
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int i = ctid + it * kConvThreads;
    if (i < kGroups) {
      const int j = i >> 4, k = i & 15;
      const int32_t sr = src[tt * kRows + j];
      unsigned char* dst = xc + j * 256 + k * 16;
      if (sr >= 0) {
        if (k < ng) cp_async16(dst, nope + static_cast<int64_t>(sr) * a.d_nope + c * 128 + k * 16);
        else if (k < ng + ngr) cp_async16(dst, rope + static_cast<int64_t>(sr) * a.d_rope + cs.rope0 + (k - ng) * 8);
      } else if (sr <= -2) {
        cp_async16(dst, win + (static_cast<int64_t>(b) * a.window + (-2 - sr)) * a.D + c * 128 + k * 8);
      }
    }
  }
}

// Convert chunk c of tile tt in place: every converter thread first reads the
// raw bytes of its 8-dim groups (group i: row i / 16, dims 8 * (i % 16) of the
// chunk), then, after a barrier of the converter group, writes them as f16 into
// the two 64-dim swizzle atoms of the chunk. Tracks the largest |value| that
// must fit f16 (range check).
DSV4_DEV void convert_chunk(const AttnArgs& a, const int32_t* src, const float* sc, int tt, int c,
                            unsigned char* xc, int ctid, float& mx) {
  const ChunkSplit cs = chunk_split(a, c);
  uint4 raw[kItems];
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int i = ctid + it * kConvThreads;
    raw[it] = make_uint4(0u, 0u, 0u, 0u);
    if (i < kGroups) {
      const int j = i >> 4, g = i & 15;
      const int32_t sr = src[tt * kRows + j];
      const unsigned char* row = xc + j * 256;
      if (sr >= 0) {
        if (8 * g < cs.nn) {
          const uint2 w = *reinterpret_cast<const uint2*>(row + 8 * g);
          raw[it].x = w.x;
          raw[it].y = w.y;
        } else {
          raw[it] = *reinterpret_cast<const uint4*>(row + cs.nn + 2 * (8 * g - cs.nn));
        }
      } else if (sr <= -2) {
        raw[it] = *reinterpret_cast<const uint4*>(row + 16 * g);
      }
    }
  }
  tc::bar_named(kBarConv, kConvThreads);
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int i = ctid + it * kConvThreads;
    if (i < kGroups) {
      const int j = i >> 4, g = i & 15;
      const int32_t sr = src[tt * kRows + j];
      uint4 h;
      if (sr >= 0 && 8 * g < cs.nn) {   // e4m3 codes times the row's scale
        const float scl = sc[tt * kRows + j];
        mx = fmaxf(mx, fabsf(scl) * 448.f);
        uint32_t s2;
        asm("{\n.reg .b16 t;\ncvt.rn.f16.f32 t, %1;\nmov.b32 %0, {t, t};\n}" : "=r"(s2) : "f"(scl * 256.f));
        h = make_uint4(e4m3x2_to_f16x2_scaled(raw[it].x, 0x4140u, s2), e4m3x2_to_f16x2_scaled(raw[it].x, 0x4342u, s2),
                       e4m3x2_to_f16x2_scaled(raw[it].y, 0x4140u, s2), e4m3x2_to_f16x2_scaled(raw[it].y, 0x4342u, s2));
      } else {
        h = bf16x8_to_f16x8(raw[it], mx);
      }
      const int atom = g >> 3, gg = g & 7;
      *reinterpret_cast<uint4*>(xc + atom * kAtomBytes + j * 128 + ((gg ^ (j & 7)) << 4)) = h;
    }
  }
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

// 32 scores (heads [col, col + 32)) of this thread's row, scaled to the log2
// domain; -inf for a row that does not exist.
DSV4_DEV void load_scores32(uint32_t taddr, float c2, bool valid, float* s) {
  uint32_t v[32];
  tc::tmem_ld32(taddr, v);
  tc::tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) s[i] = valid ? __uint_as_float(v[i]) * c2 : -INFINITY;
}

}  // namespace

// grid (splits, B, head groups), block 512. See the top of the file.
template <bool SEP>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int D = a.D;
  const int nch = D / 128;
  unsigned char* qs = base;                                  // D/64 atoms of [64 heads][128 B]
  unsigned char* pb = qs + D * 128;                          // [128 rows][64 heads] f16
  unsigned char* xk = pb + kPBytes;                          // nch chunks of [2 atoms][128 rows][128 B]
  unsigned char* xv = SEP ? xk + nch * kChunkBytes : xk;
  uint16_t* stage16 = reinterpret_cast<uint16_t*>(xk);      // epilogue: [D][64 heads] f16, after the last P.V
  const int xbytes = (SEP ? 2 : 1) * nch * kChunkBytes;
  unsigned char* qstage = xk + xbytes - 128 * D;             // prologue: raw bf16 query [64][D], top of X
  TcTail* t = reinterpret_cast<TcTail*>(xk + (SEP ? 2 : 1) * nch * kChunkBytes);
  pdl_trigger();
  pdl_wait();

  const int split = blockIdx.x, b = blockIdx.y;
  const int h0 = blockIdx.z * kHeads;
  const int hcount = a.H - h0 < kHeads ? a.H - h0 : kHeads;
  const RowSpace rs = row_space(a, b);
  const int64_t r0 = static_cast<int64_t>(split) * a.rows_per_split;
  const int64_t r1 = r0 + a.rows_per_split < rs.R ? r0 + a.rows_per_split : rs.R;
  const int nt = r1 > r0 ? static_cast<int>((r1 - r0 + kRows - 1) / kRows) : 0;
  if (nt == 0) {   // uniform: nothing to attend in this split
    for (int h = threadIdx.x; h < hcount; h += blockDim.x)
      a.part_lse[(static_cast<int64_t>(b) * a.H + h0 + h) * a.splits + split] = -INFINITY;
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(kHeads * (1 + nch))) cols <<= 1;
  volatile int* abort = &t->abort;
  const int nrows = nt * kRows;   // <= kMaxTiles * kRows (host plan)

  if (a.n_sel == 0 && warp == 0) prefetch_rows(a, rs, b, r0, r1, SEP, lane);   // HCA: known ranges, start now
  if (warp == 0) tc::tmem_alloc(&t->taddr, cols);
  if (threadIdx.x == 32) {
    for (int c = 0; c < kMaxChunks; ++c) {
      tc::mbar_init(&t->xfull[c], kConvThreads / 32);
      tc::mbar_init(&t->xfree[c], 1);
    }
    tc::mbar_init(&t->sfull, 1);
    tc::mbar_init(&t->pfull, kSoftThreads / 32);
    tc::mbar_init(&t->pvdone, 1);
    tc::mbar_init(&t->qready, kSoftThreads / 32);
    tc::mbar_init(&t->qraw, 1);
    tc::mbar_init(&t->drain, 1);
    t->abort = 0;
    tc::fence_mbar_init();
    // the query rows of this head group, raw bf16, into the top of the X region
    const uint32_t qbytes = static_cast<uint32_t>(hcount) * D * 2;
    tc::mbar_arrive_expect_tx(&t->qraw, qbytes);
    tc::bulk_load(qstage, a.q + (static_cast<int64_t>(b) * a.H + h0) * D, qbytes, &t->qraw);
  }
  if (threadIdx.x < kHeads) t->m_used[threadIdx.x] = -INFINITY;
  {
    // row sources of the whole split (CSA: one round trip for the top-k indices)
    int32_t sr[2];
    float ks[2], vs[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = threadIdx.x + k * kThreads;
      sr[k] = i < nrows ? row_source(a, rs, b, r0 + i, r1, true) : -1;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      ks[k] = sr[k] >= 0 ? __ldg(a.k_scale + sr[k]) : 0.f;
      vs[k] = SEP && sr[k] >= 0 ? __ldg(a.v_scale + sr[k]) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = threadIdx.x + k * kThreads;
      if (i < nrows) {
        t->src[i] = sr[k];
        t->sk[i] = ks[k];
        if (SEP) t->sv[i] = vs[k];
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t taddr = t->taddr;
  const uint32_t s_tmem = taddr, o_tmem = taddr + kHeads;
  const int32_t* src = t->src;
  if (a.n_sel > 0 && warp == 0) {   // CSA: prefetch the selected rows and the window, now that they are known
    for (int i = lane; i < nrows; i += 32) {
      const int32_t sr = src[i];
      if (sr >= 0) {
        tc::prefetch_l2_bulk(a.k_nope + static_cast<int64_t>(sr) * a.d_nope, a.d_nope);
        if (a.d_rope) tc::prefetch_l2_bulk(a.k_rope + static_cast<int64_t>(sr) * a.d_rope, a.d_rope * 2);
        if (SEP) {
          tc::prefetch_l2_bulk(a.v_nope + static_cast<int64_t>(sr) * a.d_nope, a.d_nope);
          if (a.d_rope) tc::prefetch_l2_bulk(a.v_rope + static_cast<int64_t>(sr) * a.d_rope, a.d_rope * 2);
        }
      }
    }
    if (lane < (SEP ? 4 : 2)) prefetch_rows(a, rs, b, r0 > rs.n_main ? r0 : rs.n_main, r1, SEP, lane);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_f16_f32(kRows, kHeads, 0, 0);
      const uint32_t id_pv = tc::idesc_f16_f32(kRows, kHeads, 1, 1);
      const uint32_t q_sa = tc::smem_u32(qs), p_sa = tc::smem_u32(pb);
      const uint32_t xk_sa = tc::smem_u32(xk), xv_sa = tc::smem_u32(xv);
      bool ok = tc::mbar_wait(&t->qready, 0, abort);
      for (int tt = 0; ok && tt < nt; ++tt) {
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
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad =
                tc::smem_desc_lbo(xv_sa + c * kChunkBytes + kk * 2048, kAtomBytes, 1024, tc::kSwizzle128B);
            const uint64_t bd = tc::smem_desc_lbo(p_sa + kk * 2048, kAtomBytes, 1024, tc::kSwizzle128B);
            tc::mma_f16(o_tmem + c * kHeads, ad, bd, id_pv, (tt | kk) ? 1u : 0u);
          }
          tc::tc_commit(&t->xfree[c]);
        }
        tc::tc_commit(&t->pvdone);
      }
      // every MMA issued must finish before tensor memory is released
      tc::tc_commit(&t->drain);
      tc::mbar_wait_drain(&t->drain, 0);
    }
  } else if (warp < 4 || (warp >= 8 && warp < 12)) {
    // ------------------------------------------------------------ dequantisation into X
    // Per tile: the copies of every chunk are issued as soon as its X region is
    // free (all of them in flight at once), then the chunks are converted in
    // place in order. Tile 0's regions that hold the staged query wait for it.
    const int ctid = (warp < 4 ? warp - 1 : warp - 5) * 32 + lane;
    const int qoff = xbytes - 128 * D;
    float mx = 0.f;
    bool ok = true;
    for (int tt = 0; ok && tt < nt; ++tt) {
      for (int c = 0; c < nch; ++c) {
        bool w = true;
        if (tt > 0) {
          w = tc::mbar_wait(&t->xfree[c], (tt - 1) & 1, abort);
        } else {
          const int lo = c * kChunkBytes, hi_k = lo + kChunkBytes;
          const bool clash = hi_k > qoff || (SEP && lo + nch * kChunkBytes + kChunkBytes > qoff);
          if (clash) w = tc::mbar_wait(&t->qready, 0, abort);
        }
        if (!(ok = tc::bar_and(kBarConv, kConvThreads, w))) break;
        issue_chunk(a, b, src, tt, c, a.k_nope, a.k_rope, a.win_k, xk + c * kChunkBytes, ctid);
        if (SEP) issue_chunk(a, b, src, tt, c, a.v_nope, a.v_rope, a.win_v, xv + c * kChunkBytes, ctid);
        cp_async_commit();
      }
      for (int c = 0; ok && c < nch; ++c) {
        cp_async_wait(nch - 1 - c);
        tc::bar_named(kBarConv, kConvThreads);   // every thread's copies of chunk c have landed
        convert_chunk(a, src, t->sk, tt, c, xk + c * kChunkBytes, ctid, mx);
        if (SEP) {
          tc::bar_named(kBarConv, kConvThreads);
          convert_chunk(a, src, t->sv, tt, c, xv + c * kChunkBytes, ctid, mx);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&t->xfull[c]);
      }
    }
    cp_async_wait(0);
    if (mx >= kF16Max) atomicOr(a.status, DSV4_STATUS_RANGE);
  } else {
    // ------------------------------------------------------------ query, softmax, epilogue
    const int qd = warp & 3;                       // tensor-memory lane quarter
    const int hb = warp >= 12 ? 32 : 0;            // this warp's heads [hb, hb + 32)
    const int j = qd * 32 + lane;                  // row of the tile / dim of an O^T block
    const int st = (warp >= 12 ? 128 : 0) + qd * 32 + lane;   // 0..255 within the group
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const float c2 = a.sm_scale * 1.4426950408889634f;
    {
      // the query (staged raw by the bulk copy), bf16 -> f16 into the K-major
      // operand; heads beyond H zero
      const bool got = tc::bar_and(kBarSoft, kSoftThreads, tc::mbar_wait(&t->qraw, 0, abort));
      const int gpr = D / 8;   // 8-dim groups per head
      float qmax = 0.f;
      for (int i = st; got && i < kHeads * gpr; i += kSoftThreads) {
        const int h = i / gpr, d0 = (i % gpr) * 8;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (h < hcount) w = *reinterpret_cast<const uint4*>(qstage + (h * D + d0) * 2);
        const int atom = d0 >> 6, gg = (d0 >> 3) & 7;
        *reinterpret_cast<uint4*>(qs + atom * kQAtomBytes + h * 128 + ((gg ^ (h & 7)) << 4)) = bf16x8_to_f16x8(w, qmax);
      }
      if (qmax >= kF16Max) atomicOr(a.status, DSV4_STATUS_RANGE);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&t->qready);
    }
    float lw = 0.f;   // l of head hb + lane over this warp's rows
    bool ok = true;
    for (int tt = 0; tt < nt; ++tt) {
      const bool valid = src[tt * kRows + j] != -1;
      ok = tc::bar_and(kBarSoft, kSoftThreads, tc::mbar_wait(&t->sfull, tt & 1, abort));
      if (!ok) break;
      if (tt > 0) {   // the previous P.V must be done with P and O^T
        ok = tc::bar_and(kBarSoft, kSoftThreads, tc::mbar_wait(&t->pvdone, (tt - 1) & 1, abort));
        if (!ok) break;
      }
      tc::tc_fence_after();
      float s[32];
      load_scores32(s_tmem + lane_off + hb, c2, valid, s);
      bool need = false;
#pragma unroll
      for (int i = 0; i < 32; ++i) need |= s[i] > t->m_used[hb + i] + kRescale;
      if (tc::bar_or(kBarSoft, kSoftThreads, need)) {
        // the running max of some head moves: reduce this tile's column max
        warp_reduce_scatter32<true>(s, lane);
        t->red[qd][hb + lane] = s[0];
        tc::bar_named(kBarSoft, kSoftThreads);
        if (st < kHeads) {
          const float tm = fmaxf(fmaxf(t->red[0][st], t->red[1][st]), fmaxf(t->red[2][st], t->red[3][st]));
          const float mo = t->m_used[st];
          const float mn = fmaxf(mo, tm);
          t->alpha[st] = mn == -INFINITY ? 1.f : ex2(mo - mn);
          t->m_used[st] = mn;
        }
        tc::bar_named(kBarSoft, kSoftThreads);
        lw *= t->alpha[hb + lane];
        if (tt > 0) {
          for (int c = 0; c < nch; ++c) {
            uint32_t v[32];
            const uint32_t addr = o_tmem + lane_off + c * kHeads + hb;
            tc::tmem_ld32(addr, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * t->alpha[hb + i]);
            tc::tmem_st32(addr, v);
          }
          tc::tmem_wait_st();
        }
        load_scores32(s_tmem + lane_off + hb, c2, valid, s);   // the reduction consumed s
      }
      // probabilities of this row and heads, f16, into P (row j, 16-byte chunks, swizzled)
#pragma unroll
      for (int i = 0; i < 32; ++i) s[i] = valid ? ex2(s[i] - t->m_used[hb + i]) : 0.f;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int i = g * 8, gc = (hb >> 3) + g;
        *reinterpret_cast<uint4*>(pb + j * 128 + ((gc ^ (j & 7)) << 4)) =
            make_uint4(f32x2_to_f16x2(s[i], s[i + 1]), f32x2_to_f16x2(s[i + 2], s[i + 3]),
                       f32x2_to_f16x2(s[i + 4], s[i + 5]), f32x2_to_f16x2(s[i + 6], s[i + 7]));
      }
      warp_reduce_scatter32<false>(s, lane);
      lw += s[0];
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&t->pfull);
    }
    if (ok) ok = tc::mbar_wait(&t->pvdone, (nt - 1) & 1, abort);
    ok = tc::bar_and(kBarSoft, kSoftThreads, ok);
    if (ok) {
      tc::tc_fence_after();
      t->red[qd][hb + lane] = lw;
      tc::bar_named(kBarSoft, kSoftThreads);
      if (st < kHeads) {
        const float l = (t->red[0][st] + t->red[1][st]) + (t->red[2][st] + t->red[3][st]);
        t->lsum[st] = l;
        t->alpha[st] = l > 0.f ? 1.f / l : 0.f;
      }
      tc::bar_named(kBarSoft, kSoftThreads);
      // normalised O^T as f16 -> stage [D][64 heads] (this split's partial in
      // the layout of the workspace), then one bulk copy
      for (int c = 0; c < nch; ++c) {
        uint32_t v[32];
        tc::tmem_ld32(o_tmem + lane_off + c * kHeads + hb, v);
        tc::tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = f32x2_to_f16x2(__uint_as_float(v[2 * i]) * t->alpha[hb + 2 * i],
                                __uint_as_float(v[2 * i + 1]) * t->alpha[hb + 2 * i + 1]);
        uint4* dst = reinterpret_cast<uint4*>(stage16 + (c * 128 + j) * kHeads + hb);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
      }
      tc::fence_proxy_async_smem();
      tc::bar_named(kBarSoft, kSoftThreads);
      const int64_t row0 = static_cast<int64_t>(b) * a.H + h0;
      if (st == 0) {
        const int hgs = gridDim.z;
        uint16_t* part = reinterpret_cast<uint16_t*>(a.part_o) +
                         ((static_cast<int64_t>(b) * a.splits + split) * hgs + blockIdx.z) * D * kHeads;
        tc::bulk_store(part, stage16, D * kHeads * 2);
        tc::bulk_commit();
      }
      if (st < hcount) {
        const float l = t->lsum[st];
        a.part_lse[(row0 + st) * a.splits + split] =
            l > 0.f ? (t->m_used[st] + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
      if (st == 0) tc::bulk_wait();   // shared memory must outlive the copy, and its writes precede the merge
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
         sizeof(TcTail);
}

template <bool SEP>
int launch_tc(const AttnArgs& a, int head_groups, cudaStream_t st) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(attn_tc_kernel<SEP>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  const size_t smem = tc_smem_bytes(a.D, SEP);
  return launch_pdl(attn_tc_kernel<SEP>, dim3(a.splits, a.B, head_groups), dim3(kThreads), smem, st, a);
}

}  // namespace

bool attention_tc_supported(int H, int d_nope, int d_rope, int separate_v) {
  const int D = d_nope + d_rope;
  if (H < 1 || H > 128 || D % 128 || D > 128 * kMaxChunks || d_nope % 8 || d_rope % 8) return false;
  if (separate_v && D > 256) return false;
  return tc_smem_bytes(D, separate_v != 0) <= 227 * 1024;
}

int launch_attention_tc(const AttnArgs& a, int head_groups, cudaStream_t st) {
  const int e = a.separate_v ? launch_tc<true>(a, head_groups, st) : launch_tc<false>(a, head_groups, st);
  if (e) return e;
  return launch_attention_merge_tc(a, head_groups, st);
}

}  // namespace dsv4
