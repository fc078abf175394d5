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
// e_i = exp(z_i + b_i - max_i(z_i + b_i)), in fp32. An append is two kernels
// on the caller's stream: pool_append_kernel reads the old pending tokens and
// the new tokens of every block this call completes and writes its entry;
// append_tail_kernel then writes the window ring and the new pending tokens and
// advances n_tokens. Splitting them keeps the pending reads of the first
// kernel ahead of the pending writes of the second.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace dsv4 {

namespace {

// Source row of token t of sequence b: the pending plane while t < n_old,
// else the new input.
DSV4_DEV const uint16_t* token_row(const uint16_t* pend, const uint16_t* in, int b, int64_t t,
                                   int64_t n_old, int T, int ratio, int dim) {
  if (t < n_old) return pend + (static_cast<int64_t>(b) * ratio + (t % ratio)) * dim;
  return in + (static_cast<int64_t>(b) * T + (t - n_old)) * dim;
}

// Pool channels [0, dim) of one block into y (shared memory).
// x2 (optional) is a second stream gated by the same logits.
DSV4_DEV void pool_block(const AppendArgs& a, int b, int64_t j, int64_t n_old, const uint16_t* pend_x,
                         const uint16_t* in_x, const uint16_t* pend_x2, const uint16_t* in_x2,
                         const uint16_t* pend_z, const uint16_t* in_z, const float* bias, int dim,
                         float* y, float* y2) {
  const int m = a.ratio;
  for (int c = threadIdx.x; c < dim; c += blockDim.x) {
    float mx = -INFINITY;
    for (int i = 0; i < m; ++i) {
      const int64_t t = j * m + i;
      const float l = bf16_to_f32(token_row(pend_z, in_z, b, t, n_old, a.T, m, dim)[c]) + bias[i * dim + c];
      mx = fmaxf(mx, l);
    }
    float sum = 0.f, acc = 0.f, acc2 = 0.f;
    for (int i = 0; i < m; ++i) {
      const int64_t t = j * m + i;
      const float l = bf16_to_f32(token_row(pend_z, in_z, b, t, n_old, a.T, m, dim)[c]) + bias[i * dim + c];
      const float e = expf(l - mx);
      sum += e;
      acc = fmaf(e, bf16_to_f32(token_row(pend_x, in_x, b, t, n_old, a.T, m, dim)[c]), acc);
      if (y2) acc2 = fmaf(e, bf16_to_f32(token_row(pend_x2, in_x2, b, t, n_old, a.T, m, dim)[c]), acc2);
    }
    y[c] = __fdiv_rn(acc, sum);
    if (y2) y2[c] = __fdiv_rn(acc2, sum);
  }
}

// Write one pooled KV row (shared memory) as an FP8 + BF16 entry.
DSV4_DEV void store_kv_entry(const float* y, int d_nope, int d_rope, uint8_t* nope, float* scale,
                             uint16_t* rope, float* red) {
  const float s = block_quant_fp8_row(y, d_nope, nope, red);
  if (threadIdx.x == 0) *scale = s;
  for (int c = threadIdx.x; c < d_rope; c += blockDim.x) rope[c] = f32_to_bf16(y[d_nope + c]);
}

DSV4_DEV void store_fp4_row(const float* y, int cols, uint8_t* codes, uint8_t* scales) {
  for (int blk = threadIdx.x; blk < cols / 16; blk += blockDim.x)
    scales[blk] = static_cast<uint8_t>(quant_fp4_block16(y + blk * 16, codes + blk * 8));
}

}  // namespace

// grid (max blocks one call can complete, B); dynamic smem: (2*D + Di) floats + 32
__global__ void __launch_bounds__(256) pool_append_kernel(AppendArgs a) {
  extern __shared__ float smem[];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  const int D = a.d_nope + a.d_rope;
  const int m = a.ratio;
  const int64_t n_old = a.n_tokens[b];
  const int64_t n_new = n_old + a.T;
  if (n_new / m > a.capacity) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, DSV4_STATUS_CAPACITY);
    return;
  }
  const int64_t j = n_old / m + blockIdx.x;
  if ((j + 1) * m > n_new) return;
  float* yk = smem;
  float* yv = smem + D;
  float* yu = smem + 2 * D;
  float* red = yu + a.idx_dim;
  pool_block(a, b, j, n_old, a.pend_k, a.k, a.pend_v, a.v, a.pend_z, a.z, a.bias, D, yk,
             a.separate_v ? yv : nullptr);
  if (a.idx_dim) pool_block(a, b, j, n_old, a.pend_u, a.u, nullptr, nullptr, a.pend_zu, a.zu, a.bias_u,
                            a.idx_dim, yu, nullptr);
  __syncthreads();
  const int64_t e = static_cast<int64_t>(b) * a.capacity + j;
  store_kv_entry(yk, a.d_nope, a.d_rope, a.k_nope + e * a.d_nope, a.k_scale + e, a.k_rope + e * a.d_rope, red);
  if (a.separate_v)
    store_kv_entry(yv, a.d_nope, a.d_rope, a.v_nope + e * a.d_nope, a.v_scale + e, a.v_rope + e * a.d_rope, red);
  if (a.idx_dim) store_fp4_row(yu, a.idx_dim, a.idx_codes + e * (a.idx_dim / 2), a.idx_scales + e * (a.idx_dim / 16));
}

namespace {
// copy `dim` bf16 values (dim a multiple of 8, rows 16-byte aligned) with the block
DSV4_DEV void copy_row(uint16_t* dst, const uint16_t* src, int dim) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < dim / 8; i += blockDim.x) d[i] = s[i];
}
}  // namespace

// grid (B); writes the window ring and the pending tokens, then advances n_tokens.
__global__ void __launch_bounds__(256) append_tail_kernel(AppendArgs a) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int D = a.d_nope + a.d_rope;
  const int m = a.ratio;
  const int64_t n_old = a.n_tokens[b];
  const int64_t n_new = n_old + a.T;
  if (n_new / m > a.capacity) return;
  if (a.window > 0) {
    const int64_t t0 = n_new - a.window > n_old ? n_new - a.window : n_old;
    for (int64_t t = t0; t < n_new; ++t) {
      const int64_t src = static_cast<int64_t>(b) * a.T + (t - n_old);
      const int64_t dst = static_cast<int64_t>(b) * a.window + t % a.window;
      copy_row(a.win_k + dst * D, a.k + src * D, D);
      if (a.separate_v) copy_row(a.win_v + dst * D, a.v + src * D, D);
    }
  }
  if (m > 1) {
    const int64_t open = (n_new / m) * m;
    const int64_t t0 = open > n_old ? open : n_old;
    for (int64_t t = t0; t < n_new; ++t) {
      const int64_t src = static_cast<int64_t>(b) * a.T + (t - n_old);
      const int64_t dst = static_cast<int64_t>(b) * m + t % m;
      copy_row(a.pend_k + dst * D, a.k + src * D, D);
      copy_row(a.pend_z + dst * D, a.z + src * D, D);
      if (a.separate_v) copy_row(a.pend_v + dst * D, a.v + src * D, D);
      if (a.idx_dim) {
        copy_row(a.pend_u + dst * a.idx_dim, a.u + src * a.idx_dim, a.idx_dim);
        copy_row(a.pend_zu + dst * a.idx_dim, a.zu + src * a.idx_dim, a.idx_dim);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) a.n_tokens[b] = n_new;
}

// Single-token append (T = 1), grid (B), one CTA per sequence: if the token
// completes a block, pool it (old pending tokens + the new one) and store the
// entry; then write the token into the window ring and, while its block stays
// open, into the pending planes; then advance n_tokens. One CTA does all of a
// sequence's work in this order, so the pending reads precede the writes.
__global__ void __launch_bounds__(256) append_one_kernel(AppendArgs a) {
  extern __shared__ float smem[];
  pdl_trigger();
  const int b = blockIdx.x;
  const int D = a.d_nope + a.d_rope;
  {
    // The new token's rows are inputs no kernel of this library writes: their
    // 128-byte lines are pulled into L1 while the previous kernel finishes, so
    // the copies and the pooling after the wait find them there.
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
    if (p) asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
  }
  pdl_wait();
  const int m = a.ratio;
  const int64_t n_old = a.n_tokens[b];
  const int64_t n_new = n_old + 1;
  if (n_new / m > a.capacity) {
    if (threadIdx.x == 0) atomicOr(a.status, DSV4_STATUS_CAPACITY);
    return;
  }
  if (n_new % m == 0) {
    const int64_t j = n_old / m;
    float* yk = smem;
    float* yv = smem + D;
    float* yu = smem + 2 * D;
    float* red = yu + a.idx_dim;
    pool_block(a, b, j, n_old, a.pend_k, a.k, a.pend_v, a.v, a.pend_z, a.z, a.bias, D, yk,
               a.separate_v ? yv : nullptr);
    if (a.idx_dim) pool_block(a, b, j, n_old, a.pend_u, a.u, nullptr, nullptr, a.pend_zu, a.zu, a.bias_u,
                              a.idx_dim, yu, nullptr);
    __syncthreads();
    const int64_t e = static_cast<int64_t>(b) * a.capacity + j;
    store_kv_entry(yk, a.d_nope, a.d_rope, a.k_nope + e * a.d_nope, a.k_scale + e, a.k_rope + e * a.d_rope, red);
    if (a.separate_v)
      store_kv_entry(yv, a.d_nope, a.d_rope, a.v_nope + e * a.d_nope, a.v_scale + e, a.v_rope + e * a.d_rope, red);
    if (a.idx_dim)
      store_fp4_row(yu, a.idx_dim, a.idx_codes + e * (a.idx_dim / 2), a.idx_scales + e * (a.idx_dim / 16));
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

// pooling of complete blocks: grid (blocks), block 256
__global__ void __launch_bounds__(256) pool_rows_kernel(const uint16_t* x, const uint16_t* z, const float* bias,
                                                       int ratio, int dim, float* y) {
  const int64_t j = blockIdx.x;
  for (int c = threadIdx.x; c < dim; c += blockDim.x) {
    float mx = -INFINITY;
    for (int i = 0; i < ratio; ++i) mx = fmaxf(mx, bf16_to_f32(z[(j * ratio + i) * dim + c]) + bias[i * dim + c]);
    float sum = 0.f, acc = 0.f;
    for (int i = 0; i < ratio; ++i) {
      const float e = expf(bf16_to_f32(z[(j * ratio + i) * dim + c]) + bias[i * dim + c] - mx);
      sum += e;
      acc = fmaf(e, bf16_to_f32(x[(j * ratio + i) * dim + c]), acc);
    }
    y[j * dim + c] = __fdiv_rn(acc, sum);
  }
}

}  // namespace dsv4
