// Lightning indexer and top-k block selection.
//
// vibecoco.ai, "DeepSeek V4 agent architecture", section
// "混合注意力：两种压缩，交替使用": a lightning indexer running in FP4 scores the
// compressed blocks with ReLU-scored multi-head dot products and the top-k
// blocks are kept. The score of block s is
//   I_s = sum_h w_h * max(0, q_h . k_s)
// on the decoded FP4 query and key (the query is quantised with the same
// per-16 e4m3-scaled e2m1 rule as the keys). Top-k keeps the k largest scores,
// ties to the lower block index, and lists them in ascending index order.
#include "common.cuh"
#include "kernels.h"

namespace dsv4 {

// grid (B * N), block Di/16: quantise one query head to FP4 (the same rule as the
// keys) into the operand layout of the scoring MMA; padding heads (h >= Hi) get
// zero codes, zero scales and zero weight.
__global__ void quant_query_fp4_kernel(IndexArgs a) {
  const int row = blockIdx.x;               // b * N + h
  const int b = row / a.N, h = row % a.N;
  const int blk = threadIdx.x;
  const int nblk = a.Di / 16;
  if (blk >= nblk) return;
  uint8_t* codes = a.q_codes + static_cast<int64_t>(row) * (a.Di / 2) + blk * 8;
  uint8_t* scale = a.q_scales + static_cast<int64_t>(row) * nblk + blk;
  if (h >= a.Hi) {
    reinterpret_cast<uint2*>(codes)[0] = make_uint2(0u, 0u);
    *scale = 0;
  } else {
    const uint16_t* src = a.q_idx + (static_cast<int64_t>(b) * a.Hi + h) * a.Di + blk * 16;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = bf16_to_f32(src[i]);
    *scale = static_cast<uint8_t>(quant_fp4_block16(v, codes));
  }
  if (blk == 0) a.wpad[row] = h < a.Hi ? a.w[b * a.Hi + h] : 0.f;
}

namespace {
// block-wide exclusive prefix count of `flag` over 1024 threads; returns the
// prefix and stores the block total in *total (shared, read after a sync).
DSV4_DEV int block_prefix(bool flag, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    int v = warp_tot[lane];
    int incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    warp_tot[lane] = incl - v;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  const int r = warp_tot[warp] + in_warp;
  __syncthreads();
  return r;
}
}  // namespace

// grid (B), block 1024: radix select of the k-th largest score key (MSB-first,
// 8 bits a pass), then one pass in index order that keeps every key above the
// threshold and the lowest-index `need` keys equal to it.
__global__ void __launch_bounds__(1024) topk_select_kernel(IndexArgs a) {
  __shared__ int hist[256];
  __shared__ int warp_tot[32];
  __shared__ int total;
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  const int b = blockIdx.x;
  int64_t n_c = a.n_tokens[b] / a.ratio;
  if (n_c > a.capacity) n_c = a.capacity;
  const float* sc = a.scores + static_cast<int64_t>(b) * a.capacity;
  int32_t* out = a.topk + static_cast<int64_t>(b) * a.k;
  if (n_c <= a.k) {
    for (int i = threadIdx.x; i < a.k; i += blockDim.x) out[i] = i < n_c ? i : -1;
    return;
  }
  uint32_t prefix = 0, mask = 0;
  int need = a.k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (threadIdx.x < 256) hist[threadIdx.x] = 0;
    __syncthreads();
    for (int64_t s = threadIdx.x; s < n_c; s += blockDim.x) {
      const uint32_t key = score_key(sc[s]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFF], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int cum = 0, d = 255;
      for (; d > 0; --d) {
        if (cum + hist[d] >= need) break;
        cum += hist[d];
      }
      s_need = need - cum;
      s_prefix = prefix | (static_cast<uint32_t>(d) << shift);
    }
    __syncthreads();
    need = s_need;
    prefix = s_prefix;
    mask |= 0xFFu << shift;
    __syncthreads();
  }
  // prefix is now the exact key of the k-th largest score; take `need` of its ties.
  int taken = 0, ties = 0;
  for (int64_t base = 0; base < n_c; base += blockDim.x) {
    const int64_t s = base + threadIdx.x;
    const uint32_t key = s < n_c ? score_key(sc[s]) : 0u;
    const bool eq = s < n_c && key == prefix;
    const bool gt = s < n_c && key > prefix;
    const int tie_rank = ties + block_prefix(eq, warp_tot, &total);
    const int tie_total = total;
    const bool take = gt || (eq && tie_rank < need);
    const int pos = taken + block_prefix(take, warp_tot, &total);
    if (take && pos < a.k) out[pos] = static_cast<int32_t>(s);
    taken += total;
    ties += tie_total;
    __syncthreads();
  }
}

}  // namespace dsv4
