// Compressor: softmax-gated pooling along the sequence and FP8 / FP4
// quantisation of the pooled entries, plus the window ring and the open-block
// (pending) tokens.
//
// vibecoco.ai, "DeepSeek V4 agent architecture", section
// "混合注意力：两种压缩，交替使用": CSA pools every 4 tokens into one entry by
// softmax-gated pooling with a learned position bias, HCA every 128; entries
// are kept in FP8 with BF16 RoPE dims and the indexer keys in FP4.
// pnsm.cn, "DeepSeek V4 架构深度解析…", section 2.1 "CSA：压缩稀疏注意力": the
// sliding window is a ring of window_size tokens overwritten cyclically.
//
// Per block j and channel c: y[c] = sum_i e_i x_i / sum_i e_i with
// e_i = exp(z_i + b_i - max_i(z_i + b_i)), in fp32, split into the same token
// groups and summed in the same order in every kernel (pool_team, pool_slice),
// so a block's bits do not depend on how its tokens arrived. An append of T > 1
// tokens is two kernels on the caller's stream: pool_chunk_kernel (or, for
// long blocks, pool_cluster_kernel) reads the old pending tokens and the new
// tokens of every block this call completes, writes its entry and writes the
// window ring; append_tail_kernel then writes the new pending tokens and
// advances n_tokens. Splitting them keeps the pending reads of the first
// kernel ahead of the pending writes of the second. A single token is one
// kernel (append_one_kernel).
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace dsv4 {

namespace {

DSV4_DEV uint4 ld16(const uint16_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

DSV4_DEV void bf16x8(uint4 w, float* f) {
  f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xFFFF0000u);
  f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xFFFF0000u);
  f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

// Raw loads of token i's gate logits (bf16) and position bias (fp32) for the
// channels [c0, c0 + 8).
struct GateLoad {
  uint4 z;
  float4 b0, b1;
};
// the 8 logits z + b of a GateLoad
DSV4_DEV void logits8(const GateLoad& g, float* l) {
  bf16x8(g.z, l);
  l[0] += g.b0.x; l[1] += g.b0.y; l[2] += g.b0.z; l[3] += g.b0.w;
  l[4] += g.b1.x; l[5] += g.b1.y; l[6] += g.b1.z; l[7] += g.b1.w;
}

// Token rows of one compressed block j of sequence b in global memory: token
// i (0 <= i < m) is position t0 + i; positions before n_old come from the
// pending planes (slot t % m), the others from this call's inputs.
struct BlockSrc {
  const uint16_t *pend_x, *in_x, *pend_x2, *in_x2, *pend_z, *in_z;
  const float* bias;   // [m][C]
  int64_t t0, n_old;
  int b, T, m, C;
  DSV4_DEV const uint16_t* row(const uint16_t* pend, const uint16_t* in, int i) const {
    const int64_t t = t0 + i;
    return t < n_old ? pend + (static_cast<int64_t>(b) * m + (t % m)) * C
                     : in + (static_cast<int64_t>(b) * T + (t - n_old)) * C;
  }
  DSV4_DEV bool two() const { return in_x2 != nullptr; }
  DSV4_DEV GateLoad gate(int i, int c0) const {
    GateLoad g;
    g.z = ld16(row(pend_z, in_z, i) + c0);
    const float4* bp = reinterpret_cast<const float4*>(bias + static_cast<int64_t>(i) * C + c0);
    g.b0 = __ldg(bp);
    g.b1 = __ldg(bp + 1);
    return g;
  }
  DSV4_DEV uint4 x(int i, int c0) const { return ld16(row(pend_x, in_x, i) + c0); }
  DSV4_DEV uint4 x2(int i, int c0) const { return ld16(row(pend_x2, in_x2, i) + c0); }
};

// The same rows of one 64-channel slice, copied into shared memory: x, x2 (or
// null), z as [m][64] bf16 and the position bias as [m][64] fp32.
struct SmemRows {
  const uint16_t *xs, *x2s, *zs;
  const float* bs;
};

// Softmax-gated pooling of one block by a team (see PoolShape): team thread t
// takes channels [8 c8, 8 c8 + 8) and tokens [g tpg, g tpg + tpg) of the
// block, c8 = t % cg, g = t / cg. For every channel c, in fp32:
//   M = max_i (z_i + b_i)                       (exact in any order)
//   S = sum_i e_i, A = sum_i e_i x_i,  e_i = exp(z_i + b_i - M)
// each group summing its tokens in order, the groups' sums then added in
// group order; y = A / S (IEEE division). Threads of group 0 return y (and
// y2, the second stream gated by the same logits). `part` is shared memory of
// pool_part_floats() floats for this team. Every thread of the CTA calls it
// (it holds CTA barriers when G > 1); `active` marks a thread with work.
// ONE: a group's tokens fit one batch of loads (tpg <= 4), which are then all
// issued in the first pass and kept in registers for the second. The
// arithmetic, and so every result bit, is the same whatever the batching.
template <bool TWO, bool ONE>
DSV4_DEV void pool_team_t(const BlockSrc& s, PoolShape ps, int m, int t, bool active, float* part, float* y,
                          float* y2) {
  constexpr int kTokBatch = TWO ? 2 : 4;   // tokens whose loads a thread issues together
  constexpr bool two = TWO;
  const int c8 = t % ps.cg, g = t / ps.cg;
  const int c0 = 8 * c8;
  const int i0 = g * ps.tpg, i1 = i0 + ps.tpg < m ? i0 + ps.tpg : m;
  float mx[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
  GateLoad g1[ONE ? kTokBatch : 1];
  uint4 x1[ONE ? kTokBatch : 1], x21[ONE ? kTokBatch : 1];
  if (active) {
    if constexpr (ONE) {
      // the group's only batch: the gates and the values, all in flight
#pragma unroll
      for (int u = 0; u < kTokBatch; ++u)
        if (i0 + u < i1) {
          g1[u] = s.gate(i0 + u, c0);
          x1[u] = s.x(i0 + u, c0);
          if (two) x21[u] = s.x2(i0 + u, c0);
        }
#pragma unroll
      for (int u = 0; u < kTokBatch; ++u)
        if (i0 + u < i1) {
          float l[8];
          logits8(g1[u], l);
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], l[k]);
        }
    } else {
      for (int i = i0; i < i1; i += kTokBatch) {
        // a batch of tokens: every load in flight, then the maxima in token order
        GateLoad gl[kTokBatch];
#pragma unroll
        for (int u = 0; u < kTokBatch; ++u)
          if (i + u < i1) gl[u] = s.gate(i + u, c0);
#pragma unroll
        for (int u = 0; u < kTokBatch; ++u)
          if (i + u < i1) {
            float l[8];
            logits8(gl[u], l);
#pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], l[k]);
          }
      }
    }
  }
  if (ps.G > 1) {
    float* pm = part + (g * ps.cg + c8) * 8;
    if (active)
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = mx[k];
    __syncthreads();
    if (active)
      for (int h = 0; h < ps.G; ++h) {
        const float* q = part + (h * ps.cg + c8) * 8;
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], q[k]);
      }
    __syncthreads();
  }
  float sum[8], acc[8], acc2[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) sum[k] = acc[k] = acc2[k] = 0.f;
  if (active)
    for (int i = i0; i < i1; i += kTokBatch) {
      // a batch of tokens: every load in flight, then the sums in token order
      GateLoad gl[kTokBatch];
      uint4 xw[kTokBatch], x2w[kTokBatch];
#pragma unroll
      for (int u = 0; u < kTokBatch; ++u)
        if (i + u < i1) {
          if constexpr (ONE) {
            gl[u] = g1[u];
            xw[u] = x1[u];
            if (two) x2w[u] = x21[u];
          } else {
            gl[u] = s.gate(i + u, c0);
            xw[u] = s.x(i + u, c0);
            if (two) x2w[u] = s.x2(i + u, c0);
          }
        }
#pragma unroll
      for (int u = 0; u < kTokBatch; ++u)
        if (i + u < i1) {
          float l[8], x[8], x2[8];
          logits8(gl[u], l);
          bf16x8(xw[u], x);
          if (two) bf16x8(x2w[u], x2);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float e = expf(l[k] - mx[k]);
            sum[k] += e;
            acc[k] = fmaf(e, x[k], acc[k]);
            if (two) acc2[k] = fmaf(e, x2[k], acc2[k]);
          }
        }
    }
  if (ps.G > 1) {
    float* pp = part + (g * ps.cg + c8) * (two ? 24 : 16);
    if (active)
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        pp[k] = sum[k];
        pp[8 + k] = acc[k];
        if (two) pp[16 + k] = acc2[k];
      }
    __syncthreads();
    if (active && g == 0)
      for (int h = 1; h < ps.G; ++h) {
        const float* q = part + (h * ps.cg + c8) * (two ? 24 : 16);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          sum[k] += q[k];
          acc[k] += q[8 + k];
          if (two) acc2[k] += q[16 + k];
        }
      }
    __syncthreads();   // `part` is reused by the next team call
  }
  if (active && g == 0)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      y[k] = __fdiv_rn(acc[k], sum[k]);
      if (two) y2[k] = __fdiv_rn(acc2[k], sum[k]);
    }
}

// (the one-batch form for a single stream only, and where the kernel allows
// it: with two streams, or in a kernel with other work, it holds too many
// registers)
template <bool ALLOW_ONE = true>
DSV4_DEV void pool_team(const BlockSrc& s, PoolShape ps, int m, int t, bool active, float* part, float* y,
                        float* y2) {
  if (s.two()) pool_team_t<true, false>(s, ps, m, t, active, part, y, y2);
  else if (ALLOW_ONE && ps.tpg <= 4) pool_team_t<false, true>(s, ps, m, t, active, part, y, y2);   // uniform
  else pool_team_t<false, false>(s, ps, m, t, active, part, y, y2);
}

// n consecutive bf16 (n = 2, 4, 8; 4n-byte aligned) from shared memory as floats
template <int N>
DSV4_DEV void lds_bf16(const uint16_t* p, float* f) {
  if constexpr (N == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(w << 16); f[1] = __uint_as_float(w & 0xFFFF0000u);
  } else if constexpr (N == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  } else {
    bf16x8(*reinterpret_cast<const uint4*>(p), f);
  }
}

// Pooling of one block's 64-channel slice from shared memory with the team
// arithmetic of pool_team_t (G token groups of tpg tokens), the channels dealt
// CPT to a thread instead of 8, so that more threads share the same work:
// thread t takes channels [CPT q, CPT q + CPT) and tokens [g tpg, g tpg + tpg),
// q = t % (64 / CPT), g = t / (64 / CPT). Every operation on a channel is the
// one pool_team_t performs, in the same order: the same bits. Group 0's
// threads leave y (and y2) in ys[64] (ys2). `part` holds G * 64 * 3 floats.
// Every thread of the CTA calls it (CTA barriers when G > 1).
template <int CPT, bool TWO>
DSV4_DEV void pool_slice(const SmemRows& s, int G, int tpg, int m, int t, float* part, float* ys, float* ys2) {
  constexpr int NQ = 64 / CPT;
  constexpr int S = TWO ? 3 : 2;   // combined sums per channel
  const int q = t % NQ, g = t / NQ;
  const bool active = g < G;
  const int c0 = q * CPT;
  const int i0 = g * tpg, i1 = i0 + tpg < m ? i0 + tpg : m;
  float mx[CPT];
#pragma unroll
  for (int k = 0; k < CPT; ++k) mx[k] = -INFINITY;
  if (active)
    for (int i = i0; i < i1; ++i) {
      float l[CPT];
      lds_bf16<CPT>(s.zs + i * 64 + c0, l);
#pragma unroll
      for (int k = 0; k < CPT; ++k) mx[k] = fmaxf(mx[k], l[k] + s.bs[i * 64 + c0 + k]);
    }
  if (G > 1) {
    if (active)
#pragma unroll
      for (int k = 0; k < CPT; ++k) part[g * 64 + c0 + k] = mx[k];
    __syncthreads();
    if (active)
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int k = 0; k < CPT; ++k) mx[k] = fmaxf(mx[k], part[h * 64 + c0 + k]);
    __syncthreads();
  }
  float sum[CPT], acc[CPT], acc2[CPT];
#pragma unroll
  for (int k = 0; k < CPT; ++k) sum[k] = acc[k] = acc2[k] = 0.f;
  if (active)
    for (int i = i0; i < i1; ++i) {
      float l[CPT], x[CPT], x2[CPT];
      lds_bf16<CPT>(s.zs + i * 64 + c0, l);
      lds_bf16<CPT>(s.xs + i * 64 + c0, x);
      if (TWO) lds_bf16<CPT>(s.x2s + i * 64 + c0, x2);
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        const float e = expf((l[k] + s.bs[i * 64 + c0 + k]) - mx[k]);
        sum[k] += e;
        acc[k] = fmaf(e, x[k], acc[k]);
        if (TWO) acc2[k] = fmaf(e, x2[k], acc2[k]);
      }
    }
  if (G > 1) {
    if (active)
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        float* pp = part + (g * 64 + c0 + k) * S;
        pp[0] = sum[k];
        pp[1] = acc[k];
        if (TWO) pp[2] = acc2[k];
      }
    __syncthreads();
    if (active && g == 0)
      for (int h = 1; h < G; ++h)
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
          const float* pq = part + (h * 64 + c0 + k) * S;
          sum[k] += pq[0];
          acc[k] += pq[1];
          if (TWO) acc2[k] += pq[2];
        }
    __syncthreads();
  }
  if (active && g == 0)
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
      ys[c0 + k] = __fdiv_rn(acc[k], sum[k]);
      if (TWO) ys2[c0 + k] = __fdiv_rn(acc2[k], sum[k]);
    }
}


// The FP8 + BF16 entry of a pooled row held by a team's group-0 threads (8
// channels each, `has` when the thread holds some): scale = amax/448 over the
// d_nope FP8 dims, codes = e4m3(y / scale), the RoPE dims bf16.
// entry_amax: this thread's share of amax (0 when it holds no FP8 dims).
DSV4_DEV float entry_amax(const float* y, bool has, int c8, int d_nope) {
  float m = 0.f;
  if (has && 8 * c8 < d_nope)
#pragma unroll
    for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(y[k]));
  return m;
}
// entry_write: this thread's dims of the entry, given the row's amax.
DSV4_DEV void entry_write(const float* y, bool has, int c8, int d_nope, float amax, uint8_t* nope, float* scale,
                          uint16_t* rope) {
  const int c0 = 8 * c8;
  if (has && c0 < d_nope) {
    const float s = __fdiv_rn(amax, 448.f);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (s > 0.f)
#pragma unroll
      for (int k = 0; k < 4; ++k) w[k] = f32x2_to_e4m3x2(__fdiv_rn(y[2 * k], s), __fdiv_rn(y[2 * k + 1], s));
    *reinterpret_cast<uint2*>(nope + c0) = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
    if (c8 == 0) *scale = s;
  } else if (has) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = static_cast<uint32_t>(f32_to_bf16(y[2 * k])) | (static_cast<uint32_t>(f32_to_bf16(y[2 * k + 1])) << 16);
    *reinterpret_cast<uint4*>(rope + (c0 - d_nope)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
// The whole entry by one CTA: amax combined through the shared word *amax
// (zeroed by the caller before a barrier). Every thread of the CTA calls it
// (one CTA barrier).
DSV4_DEV void store_entry(const float* y, bool has, int c8, int d_nope, uint32_t* amax, uint8_t* nope, float* scale,
                          uint16_t* rope) {
  if (has && 8 * c8 < d_nope) atomicMax(amax, __float_as_uint(entry_amax(y, has, c8, d_nope)));
  __syncthreads();
  entry_write(y, has, c8, d_nope, __uint_as_float(*amax), nope, scale, rope);
}

// The FP4 row of a pooled indexer key held by a team's group-0 threads: per
// 16 channels (a pair of threads, c8 even and odd, neighbours in a warp)
// scale = e4m3(amax/6), codes = e2m1(y / scale). Every thread of the CTA calls
// it (one full-warp shuffle; a pair never spans two teams since cg is even).
DSV4_DEV void store_fp4(const float* y, bool has, int c8, uint8_t* codes, uint8_t* scales) {
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(y[k]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  if (!has) return;
  const uint32_t sc = f32_to_e4m3(__fdiv_rn(m, 6.f));
  const float s = e4m3_to_f32(sc);
  float q[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) q[k] = s > 0.f ? __fdiv_rn(y[k], s) : 0.f;
  *reinterpret_cast<uint32_t*>(codes + 4 * c8) = s > 0.f ? f32x8_to_e2m1x8(q) : 0u;
  if ((c8 & 1) == 0) scales[c8 >> 1] = static_cast<uint8_t>(sc);
}

}  // namespace

namespace {
// Copy rows of bf16 values (dim a multiple of 8, rows 16-byte aligned) with the
// whole CTA: row r of `rows` goes from src + src_row(r) * dim to dst +
// dst_row(r) * dim; every 16-byte piece is an independent item, loaded in
// groups of four before they are stored.
template <typename SrcRow, typename DstRow>
DSV4_DEV void copy_rows(uint16_t* dst, const uint16_t* src, int rows, int dim, SrcRow src_row, DstRow dst_row) {
  const int per = dim / 8;
  const int n = rows * per;
  for (int i0 = threadIdx.x; i0 < n; i0 += 4 * blockDim.x) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n) v[u] = __ldg(reinterpret_cast<const uint4*>(src + src_row(i / per) * dim) + i % per);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n) reinterpret_cast<uint4*>(dst + dst_row(i / per) * dim)[i % per] = v[u];
    }
  }
}
}  // namespace

// Pooling of every block an append of T > 1 tokens completes, and the window
// ring, grid (CTAs, B): CTAs [0, ctas_k) pool the key (and value) stream,
// bpc_k blocks per CTA (a team per block, see PoolShape), and store FP8
// entries; the next ctas_u pool the indexer-key stream, bpc_u blocks per CTA,
// and store FP4 keys; the rest write the call's last min(W, T) tokens into the
// window ring, kWinRowsPerCta rows each (no kernel reads the ring during an
// append). Dynamic shared memory: the teams' combine buffers, then one amax
// word per block.
__global__ void __launch_bounds__(512) pool_chunk_kernel(AppendArgs a) {
  extern __shared__ float smem[];
  pdl_trigger();
  const int b = blockIdx.y;
  const int D = a.d_nope + a.d_rope;
  const int m = a.ratio;
  if (threadIdx.x == 0 && static_cast<int>(blockIdx.x) < a.ctas_k + a.ctas_u) {
    // While the previous kernel finishes: the input rows this CTA pools when
    // the call starts on a block boundary (the usual case) are pulled into L2.
    // A hint only, and L2 is coherent with whatever that kernel still writes.
    const bool key_stream = static_cast<int>(blockIdx.x) < a.ctas_k;
    const int bpc = key_stream ? a.bpc_k : a.bpc_u;
    const int64_t r0 = static_cast<int64_t>(key_stream ? blockIdx.x : blockIdx.x - a.ctas_k) * bpc * m;
    const int64_t r1 = r0 + static_cast<int64_t>(bpc) * m < a.T ? r0 + static_cast<int64_t>(bpc) * m : a.T;
    if (r0 < r1) {
      const int64_t row = static_cast<int64_t>(b) * a.T + r0;
      if (key_stream) {
        tc::prefetch_l2_range(a.k + row * D, (r1 - r0) * D * 2);
        tc::prefetch_l2_range(a.z + row * D, (r1 - r0) * D * 2);
        if (a.separate_v) tc::prefetch_l2_range(a.v + row * D, (r1 - r0) * D * 2);
      } else {
        tc::prefetch_l2_range(a.u + row * a.idx_dim, (r1 - r0) * a.idx_dim * 2);
        tc::prefetch_l2_range(a.zu + row * a.idx_dim, (r1 - r0) * a.idx_dim * 2);
      }
    }
  }
  pdl_wait();
  const int64_t n_old = a.n_tokens[b];
  const int64_t n_new = n_old + a.T;
  if (n_new / m > a.capacity) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, DSV4_STATUS_CAPACITY);
    return;
  }
  if (static_cast<int>(blockIdx.x) >= a.ctas_k + a.ctas_u) {
    // window rows: tokens [n_new - cnt, n_new), cnt = min(W, T)
    const int cnt = a.T < a.window ? a.T : a.window;
    const int r0 = (blockIdx.x - a.ctas_k - a.ctas_u) * kWinRowsPerCta;
    const int rows = cnt - r0 < kWinRowsPerCta ? cnt - r0 : kWinRowsPerCta;
    if (rows <= 0) return;
    const int64_t t0 = n_new - cnt + r0;   // position of the CTA's first row
    auto src_row = [&](int r) { return static_cast<int64_t>(b) * a.T + (t0 + r - n_old); };
    auto dst_row = [&](int r) { return static_cast<int64_t>(b) * a.window + (t0 + r) % a.window; };
    copy_rows(a.win_k, a.k, rows, D, src_row, dst_row);
    if (a.separate_v) copy_rows(a.win_v, a.v, rows, D, src_row, dst_row);
    return;
  }
  const int64_t j0 = n_old / m, j1 = n_new / m;   // blocks [j0, j1) complete in this call
  const bool key_stream = static_cast<int>(blockIdx.x) < a.ctas_k;
  const int C = key_stream ? D : a.idx_dim;
  const int bpc = key_stream ? a.bpc_k : a.bpc_u;
  const PoolShape ps = pool_shape(m, C);
  const int team = ps.G * ps.cg;
  const int slot = threadIdx.x / team, t = threadIdx.x % team;
  const int64_t j = j0 + static_cast<int64_t>(key_stream ? blockIdx.x : blockIdx.x - a.ctas_k) * bpc + slot;
  const bool active = slot < bpc && j < j1;
  const bool two = key_stream && a.separate_v;
  float* part = smem + slot * pool_part_floats(ps, two);
  uint32_t* amax = reinterpret_cast<uint32_t*>(smem + bpc * pool_part_floats(ps, two)) + 2 * slot;
  if (t < 2 && slot < bpc) amax[t] = 0u;
  BlockSrc src;
  src.t0 = j * m; src.n_old = n_old; src.b = b; src.T = a.T; src.m = m; src.C = C;
  if (key_stream) {
    src.pend_x = a.pend_k; src.in_x = a.k; src.pend_x2 = a.pend_v; src.in_x2 = two ? a.v : nullptr;
    src.pend_z = a.pend_z; src.in_z = a.z; src.bias = a.bias;
  } else {
    src.pend_x = a.pend_u; src.in_x = a.u; src.pend_x2 = nullptr; src.in_x2 = nullptr;
    src.pend_z = a.pend_zu; src.in_z = a.zu; src.bias = a.bias_u;
  }
  float y[8] = {}, y2[8] = {};
  pool_team(src, ps, m, t, active, part, y, y2);
  __syncthreads();   // the amax words are zeroed
  const bool has = active && t < ps.cg;
  const int64_t e = static_cast<int64_t>(b) * a.capacity + j;
  if (key_stream) {
    store_entry(y, has, t, a.d_nope, amax, a.k_nope + e * a.d_nope, a.k_scale + e, a.k_rope + e * a.d_rope);
    if (two)
      store_entry(y2, has, t, a.d_nope, amax + 1, a.v_nope + e * a.d_nope, a.v_scale + e, a.v_rope + e * a.d_rope);
  } else {
    // every thread (whole warps: the pair shuffle; a pair never spans two teams)
    store_fp4(y, has, t, a.idx_codes + e * (a.idx_dim / 2), a.idx_scales + e * (a.idx_dim / 16));
  }
}

// Pooling of the key (and value) stream of an append of T > 1 tokens for a
// layer with blocks of more than 8 tokens, D = d_nope + d_rope a multiple of 64
// up to 512, and no indexer. Grid (ctas_k + window CTAs, B) in clusters of
// cs = D / 64 CTAs: cluster q pools block j0 + q, its CTA r the channels
// [64 r, 64 r + 64). A CTA copies the block's rows of its slice (pending
// tokens or this call's), gate logits and position bias into shared memory
// (cp.async, one round trip), pools them with the team arithmetic of every
// other pooling kernel (G token groups; 64 / CPT x G threads, CPT channels a
// thread: pool_slice, the same bits), and the cluster combines the FP8
// scale's amax in distributed shared memory before each CTA writes its dims
// of the entry. CTAs past ctas_k (whole clusters) write the window ring as
// pool_chunk_kernel does. Dynamic shared memory: bias [m][64] fp32, z, x (, v)
// [m][64] bf16, the combine buffer, four words (the cluster's amax of K and V,
// which the peers raise; this CTA's), the pooled slice (K, V) [2][64] fp32.
__global__ void __launch_bounds__(256, 1) pool_cluster_kernel(AppendArgs a) {
  extern __shared__ __align__(16) unsigned char csm[];
  const int D = a.d_nope + a.d_rope;
  const int m = a.ratio;
  const bool two = a.separate_v != 0;
  const PoolShape pk = pool_shape(m, D);
  PoolShape ps;   // the team of one 64-channel slice
  ps.cg = 8; ps.G = pk.G; ps.tpg = pk.tpg;
  float* bias_s = reinterpret_cast<float*>(csm);
  uint16_t* z_s = reinterpret_cast<uint16_t*>(bias_s + m * 64);
  uint16_t* x_s = z_s + m * 64;
  uint16_t* x2_s = x_s + m * 64;
  float* part = reinterpret_cast<float*>(x_s + (two ? 2 : 1) * m * 64);
  uint32_t* words = reinterpret_cast<uint32_t*>(part + pool_part_floats(ps, two));
  pdl_trigger();
  const int b = blockIdx.y;
  const uint32_t r = tc::cluster_rank(), cs = tc::cluster_ctas();
  const int cbase = 64 * static_cast<int>(r);
  const bool pool = static_cast<int>(blockIdx.x) < a.ctas_k;
  if (pool) {
    // the slice's position bias: a caller input that no kernel of this library writes
    for (int i = threadIdx.x; i < m * 16; i += blockDim.x)
      tc::cp_async16(bias_s + (i >> 4) * 64 + (i & 15) * 4, a.bias + static_cast<int64_t>(i >> 4) * D + cbase + (i & 15) * 4);
    tc::cp_async_commit();
    // the input rows of the cluster's block when the call starts on a block
    // boundary (the usual case), this CTA's share of them, into L2: a hint
    // only, and L2 is coherent with whatever the previous kernel still writes
    const int64_t i0 = static_cast<int64_t>(blockIdx.x / cs) * m;
    const int64_t i1 = i0 + m < a.T ? i0 + m : a.T;
    const int64_t share = (i1 - i0 + cs - 1) / cs;
    const int64_t r0 = i0 + r * share, r1 = r0 + share < i1 ? r0 + share : i1;
    if (threadIdx.x == 0 && r0 < r1) {
      const int64_t row = static_cast<int64_t>(b) * a.T + r0;
      tc::prefetch_l2_range(a.z + row * D, (r1 - r0) * D * 2);
      tc::prefetch_l2_range(a.k + row * D, (r1 - r0) * D * 2);
      if (two) tc::prefetch_l2_range(a.v + row * D, (r1 - r0) * D * 2);
    }
  }
  if (threadIdx.x < 4) words[threadIdx.x] = 0u;
  tc::cluster_arrive();   // the amax words are zeroed before any peer raises them
  pdl_wait();
  const int64_t n_old = a.n_tokens[b];
  const int64_t n_new = n_old + a.T;
  const int64_t j = n_old / m + static_cast<int64_t>(blockIdx.x / cs);   // the cluster's block
  bool work = pool && j < n_new / m;                                   // uniform across a cluster
  if (n_new / m > a.capacity) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, DSV4_STATUS_CAPACITY);
    work = false;
  } else if (!pool) {
    // window rows: tokens [n_new - cnt, n_new), cnt = min(W, T)
    const int cnt = a.T < a.window ? a.T : a.window;
    const int r0 = (blockIdx.x - a.ctas_k) * kWinRowsPerCta;
    const int rows = cnt - r0 < kWinRowsPerCta ? cnt - r0 : kWinRowsPerCta;
    if (rows > 0) {
      const int64_t t0 = n_new - cnt + r0;
      auto src_row = [&](int q) { return static_cast<int64_t>(b) * a.T + (t0 + q - n_old); };
      auto dst_row = [&](int q) { return static_cast<int64_t>(b) * a.window + (t0 + q) % a.window; };
      copy_rows(a.win_k, a.k, rows, D, src_row, dst_row);
      if (two) copy_rows(a.win_v, a.v, rows, D, src_row, dst_row);
    }
  }
  if (!work) {
    tc::cp_async_wait_all();   // no copy may land after the CTA has gone
    tc::cluster_wait();
    return;
  }
  BlockSrc src;
  src.t0 = j * m; src.n_old = n_old; src.b = b; src.T = a.T; src.m = m; src.C = D;
  src.pend_x = a.pend_k; src.in_x = a.k; src.pend_x2 = a.pend_v; src.in_x2 = two ? a.v : nullptr;
  src.pend_z = a.pend_z; src.in_z = a.z; src.bias = a.bias;
  for (int i = threadIdx.x; i < m * 8; i += blockDim.x) {
    const int row = i >> 3, q = (i & 7) * 8;
    tc::cp_async16(z_s + row * 64 + q, src.row(src.pend_z, src.in_z, row) + cbase + q);
    tc::cp_async16(x_s + row * 64 + q, src.row(src.pend_x, src.in_x, row) + cbase + q);
    if (two) tc::cp_async16(x2_s + row * 64 + q, src.row(src.pend_x2, src.in_x2, row) + cbase + q);
  }
  tc::cp_async_commit();
  tc::cp_async_wait_all();
  __syncthreads();
  SmemRows rows;
  rows.xs = x_s; rows.x2s = two ? x2_s : nullptr; rows.zs = z_s; rows.bs = bias_s;
  const int t = threadIdx.x;
  float* ys = reinterpret_cast<float*>(words + 4);   // the pooled slice [64] (and V's [64])
  switch (slice_cpt(ps.G) * (two ? -1 : 1)) {       // uniform across the CTA
    case 2: pool_slice<2, false>(rows, ps.G, ps.tpg, m, t, part, ys, ys + 64); break;
    case 4: pool_slice<4, false>(rows, ps.G, ps.tpg, m, t, part, ys, ys + 64); break;
    case 8: pool_slice<8, false>(rows, ps.G, ps.tpg, m, t, part, ys, ys + 64); break;
    case -2: pool_slice<2, true>(rows, ps.G, ps.tpg, m, t, part, ys, ys + 64); break;
    case -4: pool_slice<4, true>(rows, ps.G, ps.tpg, m, t, part, ys, ys + 64); break;
    default: pool_slice<8, true>(rows, ps.G, ps.tpg, m, t, part, ys, ys + 64); break;
  }
  __syncthreads();
  // the entry's dims, 8 to a thread as every other pooling kernel writes them
  const bool has = t < 8;
  float y[8] = {}, y2[8] = {};
  if (has)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      y[k] = ys[8 * t + k];
      y2[k] = ys[64 + 8 * t + k];
    }
  const int c8 = cbase / 8 + t;   // the thread's channel group in the row
  if (has && 8 * c8 < a.d_nope) {
    atomicMax(&words[2], __float_as_uint(entry_amax(y, has, c8, a.d_nope)));
    if (two) atomicMax(&words[3], __float_as_uint(entry_amax(y2, has, c8, a.d_nope)));
  }
  __syncthreads();
  tc::cluster_wait();   // every CTA of the cluster has zeroed its amax words
  if (threadIdx.x < cs) {
    tc::peer_max(tc::peer_addr(&words[0], threadIdx.x), words[2]);
    if (two) tc::peer_max(tc::peer_addr(&words[1], threadIdx.x), words[3]);
  }
  tc::cluster_sync();   // every CTA holds the row's amax; no peer touches this CTA's memory after it
  const int64_t e = static_cast<int64_t>(b) * a.capacity + j;
  entry_write(y, has, c8, a.d_nope, __uint_as_float(words[0]), a.k_nope + e * a.d_nope, a.k_scale + e,
              a.k_rope + e * a.d_rope);
  if (two)
    entry_write(y2, has, c8, a.d_nope, __uint_as_float(words[1]), a.v_nope + e * a.d_nope, a.v_scale + e,
                a.v_rope + e * a.d_rope);
}

namespace {
// copy `dim` bf16 values (dim a multiple of 8, rows 16-byte aligned) with the block
DSV4_DEV void copy_row(uint16_t* dst, const uint16_t* src, int dim) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < dim / 8; i += blockDim.x) d[i] = s[i];
}
}  // namespace

// grid (B); after pool_chunk_kernel: writes the tokens of the block left open
// into the pending planes, then advances n_tokens.
__global__ void __launch_bounds__(256) append_tail_kernel(AppendArgs a) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int D = a.d_nope + a.d_rope;
  const int m = a.ratio;
  const int64_t n_old = a.n_tokens[b];
  const int64_t n_new = n_old + a.T;
  if (n_new / m > a.capacity) return;
  if (m > 1) {
    const int64_t open = (n_new / m) * m;
    const int64_t t0 = open > n_old ? open : n_old;   // tokens [t0, n_new) stay open
    const int rows = static_cast<int>(n_new - t0);
    auto src_row = [&](int r) { return static_cast<int64_t>(b) * a.T + (t0 + r - n_old); };
    auto dst_row = [&](int r) { return static_cast<int64_t>(b) * m + (t0 + r) % m; };
    copy_rows(a.pend_k, a.k, rows, D, src_row, dst_row);
    copy_rows(a.pend_z, a.z, rows, D, src_row, dst_row);
    if (a.separate_v) copy_rows(a.pend_v, a.v, rows, D, src_row, dst_row);
    if (a.idx_dim) {
      copy_rows(a.pend_u, a.u, rows, a.idx_dim, src_row, dst_row);
      copy_rows(a.pend_zu, a.zu, rows, a.idx_dim, src_row, dst_row);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) a.n_tokens[b] = n_new;
}

// Single-token append (T = 1), grid (B), one CTA per sequence (at least as
// many threads as the largest pooling team of the layer): if the token
// completes a block, pool it (old pending tokens + the new one) with the same
// teams as pool_chunk_kernel and store the entry; then write the token into
// the window ring and, while its block stays open, into the pending planes;
// then advance n_tokens. One CTA does all of a sequence's work in this order,
// so the pending reads precede the writes.
__global__ void __launch_bounds__(512) append_one_kernel(AppendArgs a) {
  extern __shared__ float smem[];
  pdl_trigger();
  const int b = blockIdx.x;
  const int D = a.d_nope + a.d_rope;
  {
    // The new token's 128-byte lines are pulled into L2 while the previous
    // kernel finishes, so the copies and the pooling after the wait find them
    // there. Only L2, which every SM sees coherently: the rows may be written
    // by that kernel (dsv4_project_streams), and a line held in this SM's L1
    // from before its writes would be stale.
    const int lk = D * 2 / 128, lu = a.idx_dim * 2 / 128;
    const int i = threadIdx.x;
    const char* p = nullptr;
    if (i < lk) p = reinterpret_cast<const char*>(a.k + static_cast<int64_t>(b) * D) + i * 128;
    else if (i < 2 * lk) p = reinterpret_cast<const char*>(a.z + static_cast<int64_t>(b) * D) + (i - lk) * 128;
    else if (i < 3 * lk && a.separate_v) p = reinterpret_cast<const char*>(a.v + static_cast<int64_t>(b) * D) + (i - 2 * lk) * 128;
    else if (i >= 3 * lk && i < 3 * lk + lu && a.u)
      p = reinterpret_cast<const char*>(a.u + static_cast<int64_t>(b) * a.idx_dim) + (i - 3 * lk) * 128;
    else if (i >= 3 * lk + lu && i < 3 * lk + 2 * lu && a.zu)
      p = reinterpret_cast<const char*>(a.zu + static_cast<int64_t>(b) * a.idx_dim) + (i - 3 * lk - lu) * 128;
    if (p) asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
  }
  pdl_wait();
  const int m = a.ratio;
  const int64_t n_old = a.n_tokens[b];
  const int64_t n_new = n_old + 1;
  if (n_new / m > a.capacity) {
    if (threadIdx.x == 0) atomicOr(a.status, DSV4_STATUS_CAPACITY);
    return;
  }
  if (n_new % m == 0) {   // uniform: the token completes block j
    const int64_t j = n_old / m;
    const int64_t e = static_cast<int64_t>(b) * a.capacity + j;
    uint32_t* amax = reinterpret_cast<uint32_t*>(smem);
    float* part = smem + 4;
    if (threadIdx.x < 2) amax[threadIdx.x] = 0u;
    BlockSrc src;
    src.t0 = j * m; src.n_old = n_old; src.b = b; src.T = 1; src.m = m; src.C = D;
    src.pend_x = a.pend_k; src.in_x = a.k; src.pend_x2 = a.pend_v; src.in_x2 = a.separate_v ? a.v : nullptr;
    src.pend_z = a.pend_z; src.in_z = a.z; src.bias = a.bias;
    const PoolShape pk = pool_shape(m, D);
    const int t = threadIdx.x;
    const bool act_k = t < pk.G * pk.cg;
    float y[8] = {}, y2[8] = {};
    pool_team<false>(src, pk, m, t, act_k, part, y, y2);
    __syncthreads();
    const bool has = act_k && t < pk.cg;
    store_entry(y, has, t, a.d_nope, amax, a.k_nope + e * a.d_nope, a.k_scale + e, a.k_rope + e * a.d_rope);
    if (a.separate_v)
      store_entry(y2, has, t, a.d_nope, amax + 1, a.v_nope + e * a.d_nope, a.v_scale + e, a.v_rope + e * a.d_rope);
    if (a.idx_dim) {
      src.C = a.idx_dim;
      src.pend_x = a.pend_u; src.in_x = a.u; src.pend_x2 = nullptr; src.in_x2 = nullptr;
      src.pend_z = a.pend_zu; src.in_z = a.zu; src.bias = a.bias_u;
      const PoolShape pu = pool_shape(m, a.idx_dim);
      const bool act_u = t < pu.G * pu.cg;
      pool_team<false>(src, pu, m, t, act_u, part, y, y2);
      store_fp4(y, act_u && t < pu.cg, t, a.idx_codes + e * (a.idx_dim / 2), a.idx_scales + e * (a.idx_dim / 16));
    }
    __syncthreads();
  }
  const int64_t src = b;   // row b of the [B][1][.] inputs
  if (a.window > 0) {
    const int64_t dst = static_cast<int64_t>(b) * a.window + n_old % a.window;
    copy_row(a.win_k + dst * D, a.k + src * D, D);
    if (a.separate_v) copy_row(a.win_v + dst * D, a.v + src * D, D);
  }
  if (m > 1 && n_new % m != 0) {
    const int64_t dst = static_cast<int64_t>(b) * m + n_old % m;
    copy_row(a.pend_k + dst * D, a.k + src * D, D);
    copy_row(a.pend_z + dst * D, a.z + src * D, D);
    if (a.separate_v) copy_row(a.pend_v + dst * D, a.v + src * D, D);
    if (a.idx_dim) {
      copy_row(a.pend_u + dst * a.idx_dim, a.u + src * a.idx_dim, a.idx_dim);
      copy_row(a.pend_zu + dst * a.idx_dim, a.zu + src * a.idx_dim, a.idx_dim);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) a.n_tokens[b] = n_new;
}

// one warp per row: FP8 + BF16 entry of a pooled row
__global__ void __launch_bounds__(256) quant_kv_rows_kernel(const float* y, int64_t rows, int d_nope, int d_rope,
                                                           uint8_t* nope, float* scale, uint16_t* rope) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int D = d_nope + d_rope;
  const float* row = y + r * D;
  float amax = 0.f;
  for (int c = lane; c < d_nope; c += 32) amax = fmaxf(amax, fabsf(row[c]));
  amax = warp_max(amax);
  const float s = __fdiv_rn(amax, 448.f);
  for (int c = 2 * lane; c < d_nope; c += 64) {
    uint32_t pair = 0;
    if (s > 0.f) pair = f32x2_to_e4m3x2(__fdiv_rn(row[c], s), __fdiv_rn(row[c + 1], s));
    *reinterpret_cast<uint16_t*>(nope + r * d_nope + c) = static_cast<uint16_t>(pair);
  }
  if (lane == 0) scale[r] = s;
  for (int c = lane; c < d_rope; c += 32) rope[r * d_rope + c] = f32_to_bf16(row[d_nope + c]);
}

// one thread per 16-value block
__global__ void __launch_bounds__(256) quant_fp4_rows_kernel(const float* y, int64_t rows, int cols,
                                                            uint8_t* codes, uint8_t* scales) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int per_row = cols / 16;
  if (i >= rows * per_row) return;
  const int64_t r = i / per_row;
  const int blk = static_cast<int>(i % per_row);
  float v[16];
  const float4* src = reinterpret_cast<const float4*>(y + r * cols + blk * 16);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 f = src[q];
    v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
  }
  scales[r * per_row + blk] = static_cast<uint8_t>(quant_fp4_block16(v, codes + r * (cols / 2) + blk * 8));
}

// pooling of complete blocks with the teams of the append kernels: grid
// (blocks), one team per CTA (dynamic shared memory: its combine buffer)
__global__ void __launch_bounds__(512) pool_rows_kernel(const uint16_t* x, const uint16_t* z, const float* bias,
                                                       int ratio, int dim, float* y) {
  extern __shared__ float smem[];
  const int64_t j = blockIdx.x;
  BlockSrc src;
  src.t0 = j * ratio; src.n_old = 0; src.b = 0; src.T = 0; src.m = ratio; src.C = dim;
  src.pend_x = nullptr; src.in_x = x; src.pend_x2 = nullptr; src.in_x2 = nullptr; src.pend_z = nullptr; src.in_z = z;
  src.bias = bias;
  const PoolShape ps = pool_shape(ratio, dim);
  const int t = threadIdx.x;
  float v[8] = {}, v2[8] = {};
  pool_team(src, ps, ratio, t, t < ps.G * ps.cg, smem, v, v2);
  if (t < ps.cg) {
    float4* out = reinterpret_cast<float4*>(y + j * dim + 8 * t);
    out[0] = make_float4(v[0], v[1], v[2], v[3]);
    out[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

}  // namespace dsv4
