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
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "select.cuh"

namespace dsv4 {

// grid (B * N), block Di/16: quantise one query head to FP4 (the same rule as the
// keys) into the operand layout of the scoring MMA; padding heads (h >= Hi) get
// zero codes, zero scales and zero weight.
__global__ void quant_query_fp4_kernel(IndexArgs a) {
  pdl_trigger();
  pdl_wait();
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
  // zero this sequence's top-k histograms and counters (the N blocks of a sequence share the work)
  const int words = 2 * kBins + kCntWords;
  const int per = (words + a.N - 1) / a.N;
  for (int i = h * per + blk; i < (h + 1) * per && i < words; i += nblk) {
    if (i < kBins) a.hist1[static_cast<int64_t>(b) * kBins + i] = 0;
    else if (i < 2 * kBins) a.hist2[static_cast<int64_t>(b) * kBins + (i - kBins)] = 0;
    else a.cnt[b * kCntWords + (i - 2 * kBins)] = 0;
  }
}

namespace {

constexpr int kSelThreads = 512;
constexpr int kMaxK = 2048;
constexpr int kScanItems = 8;        // scores each thread loads per round trip
constexpr int kCandCache = 4096;     // candidates the resolving CTA keeps in shared memory

// Append `flag`-ed values of a warp to list[*counter ...] with one atomic per
// warp; positions at or beyond `cap` are dropped.
DSV4_DEV void warp_append_i32(bool flag, int32_t v, uint32_t* counter, int32_t* list, uint32_t cap) {
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  if (!bal) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(bal) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(bal)));
  base = __shfl_sync(0xffffffffu, base, leader);
  const uint32_t pos = base + __popc(bal & ((1u << lane) - 1u));
  if (flag && pos < cap) list[pos] = v;
}

DSV4_DEV void warp_append_u64(bool flag, uint64_t v, uint32_t* counter, uint64_t* list, uint32_t cap) {
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  if (!bal) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(bal) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(bal)));
  base = __shfl_sync(0xffffffffu, base, leader);
  const uint32_t pos = base + __popc(bal & ((1u << lane) - 1u));
  if (flag && pos < cap) list[pos] = v;
}

// Ascending bitonic sort of the P (a power of two, <= 4 * kSelThreads) values
// of v (shared memory). With P <= kSelThreads every thread holds one value and
// strides below 32 exchange through warp shuffles.
DSV4_DEV void block_sort_asc(int32_t* v, int P) {
  const int t = threadIdx.x;
  if (P <= kSelThreads) {
    int32_t x = t < P ? v[t] : 0x7FFFFFFF;
    for (int size = 2; size <= P; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        int32_t y;
        if (stride >= 32) {
          __syncthreads();
          if (t < P) v[t] = x;
          __syncthreads();
          y = t < P ? v[t ^ stride] : 0x7FFFFFFF;
        } else {
          y = __shfl_xor_sync(0xffffffffu, x, stride);
        }
        const bool up = (t & size) == 0, lower = (t & stride) == 0;
        x = (lower == up) ? min(x, y) : max(x, y);
      }
    }
    __syncthreads();
    if (t < P) v[t] = x;
    __syncthreads();
    return;
  }
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = t; i < P / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool asc = (lo & size) == 0;
        const int32_t x = v[lo], y = v[hi];
        if ((x > y) == asc) {
          v[lo] = y;
          v[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

}  // namespace

// Top-k selection, grid (sel_ctas, B), block 512. The scoring kernel has
// histogrammed the top 12 bits of every score key and its last CTA stored the
// threshold bin T1 (the bin holding the k-th largest key) and the number of keys
// above it. Each CTA scans its slice of the scores, appends every block above
// T1 to `above` and every block in T1 to `cand` (key, index) while
// histogramming the next 12 key bits (hist2). The last CTA of the sequence to
// finish (a completion counter, no waiting) resolves the boundary: candidates
// above the second-level threshold bin are taken, the remaining ties are
// settled by the low 8 key bits and then the lower index, and the k indices are
// sorted ascending.
__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(IndexArgs a) {
  __shared__ uint32_t h[kBins];
  __shared__ int32_t fin[kMaxK];
  __shared__ uint32_t scratch[kSelThreads / 32 + 2];
  __shared__ uint32_t s_nfin, s_last, s_d, s_rem;
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  int64_t n_c = a.n_tokens[b] / a.ratio;
  if (n_c > a.capacity) n_c = a.capacity;
  int32_t* out = a.topk + static_cast<int64_t>(b) * a.k;
  const int k = a.k;
  if (n_c <= k) {
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < n_c ? i : -1;
    return;
  }
  const float* sc = a.scores + static_cast<int64_t>(b) * a.capacity;
  uint32_t* cnt = a.cnt + b * kCntWords;
  int32_t* above = a.above + static_cast<int64_t>(b) * k;
  uint64_t* cand = a.cand + static_cast<int64_t>(b) * a.capacity;
  uint32_t* hist2 = a.hist2 + static_cast<int64_t>(b) * kBins;
  const uint32_t T1 = cnt[4];   // issued with the n_tokens load above

  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int64_t chunk = (n_c + gridDim.x - 1) / gridDim.x;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * chunk;
  const int64_t c1 = c0 + chunk < n_c ? c0 + chunk : n_c;
  for (int64_t base = c0; base < c1; base += kScanItems * blockDim.x) {
    float v[kScanItems];
#pragma unroll
    for (int u = 0; u < kScanItems; ++u) {
      const int64_t s = base + threadIdx.x + u * blockDim.x;
      v[u] = s < c1 ? __ldg(sc + s) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kScanItems; ++u) {
      const int64_t s = base + threadIdx.x + u * blockDim.x;
      const bool in = s < c1;
      const uint32_t key = in ? score_key(v[u]) : 0u;
      const uint32_t bin = key >> 20;
      const bool gt = in && bin > T1;
      const bool eq = in && bin == T1;
      warp_append_i32(gt, static_cast<int32_t>(s), &cnt[0], above, static_cast<uint32_t>(k));
      warp_append_u64(eq, (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(s), &cnt[1], cand,
                      static_cast<uint32_t>(a.capacity));
      if (eq) atomicAdd(&h[(key >> 8) & 0xFFF], 1u);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kBins; i += blockDim.x)
    if (h[i]) atomicAdd(&hist2[i], h[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&cnt[2], 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- the last CTA of sequence b resolves the boundary
  uint32_t n_above = *reinterpret_cast<volatile uint32_t*>(&cnt[0]);
  uint32_t n_cand = *reinterpret_cast<volatile uint32_t*>(&cnt[1]);
  if (n_above > static_cast<uint32_t>(k)) n_above = k;                      // only on inconsistent input
  if (n_cand > static_cast<uint32_t>(a.capacity)) n_cand = a.capacity;
  const uint32_t need1 = static_cast<uint32_t>(k) - n_above;                 // taken from cand
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = reinterpret_cast<volatile uint32_t*>(hist2)[i];
  for (uint32_t i = threadIdx.x; i < n_above; i += blockDim.x) fin[i] = reinterpret_cast<volatile int32_t*>(above)[i];
  if (threadIdx.x == 0) s_nfin = n_above;
  // the candidates, read once: into shared memory when they fit
  extern __shared__ uint64_t cache[];
  const volatile uint64_t* cl = reinterpret_cast<volatile uint64_t*>(cand);
  if (n_cand <= static_cast<uint32_t>(kCandCache)) {
    for (uint32_t i0 = 0; i0 < n_cand; i0 += kScanItems * blockDim.x) {
      uint64_t v[kScanItems];
#pragma unroll
      for (int u = 0; u < kScanItems; ++u) {
        const uint32_t i = i0 + threadIdx.x + u * blockDim.x;
        v[u] = i < n_cand ? cl[i] : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kScanItems; ++u) {
        const uint32_t i = i0 + threadIdx.x + u * blockDim.x;
        if (i < n_cand) cache[i] = v[u];
      }
    }
    cl = cache;
  }
  __syncthreads();
  uint32_t n_gt2 = 0;
  const uint32_t T2 = need1 ? static_cast<uint32_t>(block_suffix_select<kSelThreads>(h, need1, &n_gt2, scratch)) : 0xFFFFu;
  const uint32_t need2 = need1 - n_gt2;                                      // taken among the keys of bin (T1, T2)
  // Candidates strictly above T2 are in; ties at (T1, T2) are ranked by the low
  // 8 key bits, then the lower index: radix select of the need2-th largest
  // 40-bit rank (low8 << 32 | ~index) among them.
  uint64_t thr_rank = 0;
  const uint32_t n_eq2 = T2 < static_cast<uint32_t>(kBins) ? h[T2] : 0u;
  if (need2 > 0 && need2 < n_eq2) {
    uint64_t prefix = 0, mask = 0;
    uint32_t remaining = need2;
    for (int pass = 0; pass < 5; ++pass) {
      const int shift = 32 - 8 * pass;                                       // bits 39..32, 31..24, ..., 7..0
      __syncthreads();
      for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
      __syncthreads();
      for (uint32_t i = threadIdx.x; i < n_cand; i += blockDim.x) {
        const uint64_t v = cl[i];
        const uint32_t key = static_cast<uint32_t>(v >> 32);
        if (((key >> 8) & 0xFFF) != T2) continue;
        const uint64_t rank = (static_cast<uint64_t>(key & 0xFF) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(v));
        if ((rank & mask) == prefix) atomicAdd(&h[(rank >> shift) & 0xFF], 1u);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        s_d = 0;
        s_rem = 0;
      }
      __syncthreads();
      if (threadIdx.x < 32) warp_digit_select(h, remaining, &s_d, &s_rem);   // s_rem: count above the digit
      __syncthreads();
      const uint32_t digit = s_d, above_digit = s_rem;
      prefix |= static_cast<uint64_t>(digit) << shift;
      mask |= static_cast<uint64_t>(0xFF) << shift;
      remaining -= above_digit;
    }
    thr_rank = prefix;                                                       // exactly need2 ranks are >= prefix
  }
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < n_cand; i += blockDim.x) {
    const uint64_t v = cl[i];
    const uint32_t key = static_cast<uint32_t>(v >> 32);
    const uint32_t b2 = (key >> 8) & 0xFFF;
    bool take = need1 > 0 && b2 > T2;
    if (b2 == T2) {
      const uint64_t rank = (static_cast<uint64_t>(key & 0xFF) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(v));
      take = need2 > 0 && (need2 >= n_eq2 || rank >= thr_rank);
    }
    if (take) {
      const uint32_t pos = atomicAdd(&s_nfin, 1u);
      if (pos < static_cast<uint32_t>(k)) fin[pos] = static_cast<int32_t>(static_cast<uint32_t>(v));
    }
  }
  __syncthreads();
  int P = 1;
  while (P < k) P <<= 1;
  for (int i = threadIdx.x + k; i < P; i += blockDim.x) fin[i] = 0x7FFFFFFF;
  __syncthreads();
  block_sort_asc(fin, P);
  for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = fin[i];
}

int launch_topk_select(const IndexArgs& a, int sel_ctas, cudaStream_t st) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kCandCache * static_cast<int>(sizeof(uint64_t)));
  });
  return launch_pdl(topk_select_kernel, dim3(sel_ctas, a.B), dim3(kSelThreads), kCandCache * sizeof(uint64_t), st, a);
}

}  // namespace dsv4
