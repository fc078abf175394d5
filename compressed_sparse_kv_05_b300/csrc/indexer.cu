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
  const int row = blockIdx.x;               // b * N + h
  const int b = row / a.N, h = row % a.N;
  const int blk = threadIdx.x;
  const int nblk = a.Di / 16;
  // the indexer query and head weights are inputs no kernel of this library
  // writes: read before the wait; every write (the workspace) after it
  const bool live = blk < nblk && h < a.Hi;
  float v[16];
  if (live) {
    const uint16_t* src = a.q_idx + (static_cast<int64_t>(b) * a.Hi + h) * a.Di + blk * 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = bf16_to_f32(src[i]);
  }
  const float wv = blk == 0 && h < a.Hi ? a.w[b * a.Hi + h] : 0.f;
  pdl_wait();
  if (blk >= nblk) return;
  uint8_t* codes = a.q_codes + static_cast<int64_t>(row) * (a.Di / 2) + blk * 8;
  uint8_t* scale = a.q_scales + static_cast<int64_t>(row) * nblk + blk;
  if (!live) {
    reinterpret_cast<uint2*>(codes)[0] = make_uint2(0u, 0u);
    *scale = 0;
  } else {
    *scale = static_cast<uint8_t>(quant_fp4_block16(v, codes));
  }
  if (blk == 0) a.wpad[row] = wv;
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
constexpr int kRegCand = 8;         // candidates per thread kept in registers by the resolving CTA
constexpr int kDigitPasses = 4;     // 8-bit index digits (indices < 2^32)
constexpr int kBitmapWords = 10240; // bitmap emission of the selection: n_c <= 327680
constexpr int kTopkDynSmem = (kCandCache * 8 > kBitmapWords * 4 ? kCandCache * 8 : kBitmapWords * 4);

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

namespace {

// Block-wide exclusive prefix sum of two 16-bit counts packed in one word
// (low: gt, high: eq); returns the exclusive prefix and writes the block total
// to *total. `scratch` holds kSelThreads / 32 words. Every thread calls it.
DSV4_DEV uint32_t block_excl_scan_packed(uint32_t v, uint32_t* total, uint32_t* scratch) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  __syncthreads();
  if (lane == 31) scratch[w] = inc;
  __syncthreads();
  uint32_t before = 0, all = 0;
  for (int ww = 0; ww < kSelThreads / 32; ++ww) {
    const uint32_t t = scratch[ww];
    if (ww < w) before += t;
    all += t;
  }
  *total = all;
  return before + inc - v;
}

// Load n words of a global array (written by other CTAs of this kernel or by
// earlier kernels) into shared memory, kScanItems loads in flight per thread.
template <typename T>
DSV4_DEV void load_to_smem(T* dst, const T* src, uint32_t n) {
  for (uint32_t i0 = 0; i0 < n; i0 += kScanItems * blockDim.x) {
    T v[kScanItems];
#pragma unroll
    for (int u = 0; u < kScanItems; ++u) {
      const uint32_t i = i0 + threadIdx.x + u * blockDim.x;
      v[u] = i < n ? __ldcg(src + i) : T(0);
    }
#pragma unroll
    for (int u = 0; u < kScanItems; ++u) {
      const uint32_t i = i0 + threadIdx.x + u * blockDim.x;
      if (i < n) dst[i] = v[u];
    }
  }
}

}  // namespace

// The resolving CTA's work when every candidate fits in registers (up to
// kRegCand per thread): T2 from the second-level histogram; inside bin
// (T1, T2) the need2 best by (low 8 key bits desc, index asc): the index
// threshold is the r-th lowest set bit of a bitmap of the tied blocks (n_c up
// to 32 * kBitmapWords), else found by 8-bit digit selections over the
// candidates held in registers; the k blocks are emitted in ascending order
// from a bitmap of the selection, else by a bitonic sort.
DSV4_DEV void resolve_in_registers(int k, int64_t n_c, uint32_t n_above, uint32_t n_cand,
                                   uint32_t need1, const uint32_t* hist2, const int32_t* above,
                                   const uint64_t* cand, int32_t* out, uint32_t* h, int32_t* fin,
                                   uint32_t (*h8)[256], uint32_t* scratch, uint64_t* dyn, uint32_t* s_nfin,
                                   uint32_t* s_d, uint32_t* s_rem) {
  const int t = threadIdx.x;
  uint64_t cv[kRegCand];
  uint32_t hv[kBins / kSelThreads];
#pragma unroll
  for (int u = 0; u < kRegCand; ++u) {
    const uint32_t i = t + u * kSelThreads;
    cv[u] = i < n_cand ? __ldcg(cand + i) : 0ull;
  }
#pragma unroll
  for (int u = 0; u < kBins / kSelThreads; ++u) hv[u] = __ldcg(hist2 + t + u * kSelThreads);
  for (uint32_t i = t; i < n_above; i += kSelThreads) fin[i] = __ldcg(above + i);
#pragma unroll
  for (int u = 0; u < kBins / kSelThreads; ++u) h[t + u * kSelThreads] = hv[u];
  for (int i = t; i < (kDigitPasses + 1) * 256; i += kSelThreads) (&h8[0][0])[i] = 0;
  if (t == 0) *s_nfin = n_above;
  __syncthreads();
  uint32_t n_gt2 = 0;
  const uint32_t T2 = need1 ? static_cast<uint32_t>(block_suffix_select<kSelThreads>(h, need1, &n_gt2, scratch)) : 0xFFFFu;
  const uint32_t need2 = need1 - n_gt2;
  const uint32_t n_eq2 = T2 < static_cast<uint32_t>(kBins) ? h[T2] : 0u;
  uint32_t d8 = 0, thr = 0;
  if (need2 > 0 && need2 < n_eq2) {
#pragma unroll
    for (int u = 0; u < kRegCand; ++u) {
      const uint32_t key = static_cast<uint32_t>(cv[u] >> 32);
      warp_hist_add(h8[0], key & 0xFF, t + u * kSelThreads < n_cand && ((key >> 8) & 0xFFF) == T2);
    }
    __syncthreads();
    if (t < 32) warp_digit_select(h8[0], need2, s_d, s_rem);
    __syncthreads();
    d8 = *s_d;
    uint32_t r = need2 - *s_rem;   // lowest indices to take among the keys with low8 == d8
    const int64_t words = (n_c + 31) / 32;
    if (r >= h8[0][d8]) {
      // every key equal to the boundary key is taken (no tie to break, the
      // usual case): no index threshold
      thr = 0xFFFFFFFFu;
    } else if (words <= kBitmapWords) {
      // the tied blocks as bits: the r-th lowest set bit is the threshold
      uint32_t* bm = reinterpret_cast<uint32_t*>(dyn);
      const int per = static_cast<int>((words + kSelThreads - 1) / kSelThreads);
      for (int i = t; i < per * kSelThreads; i += kSelThreads) bm[i] = 0;
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kRegCand; ++u) {
        const uint32_t key = static_cast<uint32_t>(cv[u] >> 32), idx = static_cast<uint32_t>(cv[u]);
        if (t + u * kSelThreads < n_cand && ((key >> 8) & 0xFFF) == T2 && (key & 0xFF) == d8)
          atomicOr(&bm[idx >> 5], 1u << (idx & 31));
      }
      __syncthreads();
      uint32_t cntw = 0;
      for (int q = 0; q < per; ++q) cntw += __popc(bm[t * per + q]);
      uint32_t tot;
      uint32_t before = block_excl_scan_packed(cntw, &tot, scratch);
      if (before < r && before + cntw >= r) {   // this thread's words hold the r-th bit
        for (int q = 0; q < per; ++q) {
          uint32_t wd = bm[t * per + q];
          const uint32_t c = __popc(wd);
          if (before + c >= r) {
            for (uint32_t k2 = r - before; k2 > 1; --k2) wd &= wd - 1;   // drop the lower set bits
            *s_d = (t * per + q) * 32 + (__ffs(wd) - 1);
            break;
          }
          before += c;
        }
      }
      __syncthreads();
      thr = *s_d;
    } else {
    int nbits = 1;
    while (nbits < 32 && (static_cast<int64_t>(1) << nbits) < n_c) ++nbits;
    const int passes = (nbits + 7) / 8;
    uint32_t prefix = 0;
    for (int p = 0; p < passes; ++p) {
      const int shift = 8 * (passes - 1 - p);
#pragma unroll
      for (int u = 0; u < kRegCand; ++u) {
        const uint32_t key = static_cast<uint32_t>(cv[u] >> 32), idx = static_cast<uint32_t>(cv[u]);
        const bool in = t + u * kSelThreads < n_cand && ((key >> 8) & 0xFFF) == T2 && (key & 0xFF) == d8 &&
                        (p == 0 || (static_cast<uint64_t>(idx) >> (shift + 8)) == prefix);
        // reversed digit: the largest reversed digit with enough keys at or above it is the smallest digit
        warp_hist_add(h8[1 + p], 255 - ((idx >> shift) & 0xFF), in);
      }
      __syncthreads();
      if (t < 32) warp_digit_select(h8[1 + p], r, s_d, s_rem);
      __syncthreads();
      prefix = (prefix << 8) | (255 - *s_d);
      r -= *s_rem;
    }
    thr = prefix;   // exactly the wanted number of indices with low8 == d8 are <= thr
    }
  }
#pragma unroll
  for (int u = 0; u < kRegCand; ++u) {
    const uint32_t key = static_cast<uint32_t>(cv[u] >> 32), idx = static_cast<uint32_t>(cv[u]);
    const uint32_t b2 = (key >> 8) & 0xFFF;
    const bool valid = t + u * kSelThreads < n_cand;
    bool take = valid && need1 > 0 && b2 > T2;
    if (valid && b2 == T2 && need2 > 0)
      take = need2 >= n_eq2 || (key & 0xFF) > d8 || ((key & 0xFF) == d8 && idx <= thr);
    warp_append_i32(take, static_cast<int32_t>(idx), s_nfin, fin, static_cast<uint32_t>(k));
  }
  __syncthreads();
  const uint32_t nf = *s_nfin < static_cast<uint32_t>(k) ? *s_nfin : static_cast<uint32_t>(k);
  const int64_t words = (n_c + 31) / 32;
  if (words <= kBitmapWords) {
    // the selected blocks as bits, then emitted in ascending order
    uint32_t* bm = reinterpret_cast<uint32_t*>(dyn);
    const int per = static_cast<int>((words + kSelThreads - 1) / kSelThreads);
    for (int i = t; i < per * kSelThreads; i += kSelThreads) bm[i] = 0;
    __syncthreads();
    for (uint32_t i = t; i < nf; i += kSelThreads) {
      const uint32_t x = static_cast<uint32_t>(fin[i]);
      atomicOr(&bm[x >> 5], 1u << (x & 31));
    }
    __syncthreads();
    uint32_t cntw = 0;
    for (int q = 0; q < per; ++q) cntw += __popc(bm[t * per + q]);
    uint32_t tot;
    const uint32_t pos = block_excl_scan_packed(cntw, &tot, scratch);
    h[t] = pos;   // set bits in the words of threads before t
    __syncthreads();
    // every selected block to its rank: set bits before it in ascending order
    for (uint32_t i = t; i < nf; i += kSelThreads) {
      const uint32_t x = static_cast<uint32_t>(fin[i]), w = x >> 5, owner = w / per;
      uint32_t r = h[owner];
      for (uint32_t v = owner * per; v < w; ++v) r += __popc(bm[v]);
      r += __popc(bm[w] & ((1u << (x & 31)) - 1u));
      if (r < static_cast<uint32_t>(k)) out[r] = static_cast<int32_t>(x);
    }
    for (uint32_t i = tot + t; i < static_cast<uint32_t>(k); i += kSelThreads) out[i] = -1;   // inconsistent input only
    return;
  }
  int P = 1;
  while (P < k) P <<= 1;
  for (int i = t + static_cast<int>(nf); i < P; i += kSelThreads) fin[i] = 0x7FFFFFFF;
  __syncthreads();
  block_sort_asc(fin, P);
  for (int i = t; i < k; i += kSelThreads) out[i] = i < static_cast<int>(nf) ? fin[i] : -1;
}

// Top-k selection, grid (sel_ctas, B), block 512. The scoring kernel has
// histogrammed the top 12 bits of every score key; every CTA finds in it the
// threshold bin T1 (the bin holding the k-th largest key). Each CTA scans its slice of the scores, appends every block above
// T1 to `above` and every block in T1 to `cand` (key, index) with one reservation
// per CTA, while histogramming the next 12 key bits (hist2). The last CTA of the
// sequence to finish (a completion counter, no waiting) resolves the boundary:
// candidates above the second-level threshold bin T2 are taken; ties in T2 are
// settled by the low 8 key bits, then by the lower index (radix select over
// 12-bit index digits); the k blocks are sorted into ascending index order.
__global__ void __launch_bounds__(kSelThreads, 2) topk_select_kernel(IndexArgs a) {
  __shared__ uint32_t h[kBins];
  __shared__ int32_t fin[kMaxK];
  __shared__ uint32_t h8[kDigitPasses + 1][256];   // resolution histograms of 8-bit digits
  __shared__ uint32_t scratch[kSelThreads / 32 + 2];
  __shared__ uint32_t s_nfin, s_last, s_d, s_rem, s_base[2];
  extern __shared__ uint64_t dyn[];   // candidate cache, or the bitmap of the selected blocks
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  // The CTA's slice of the scores is fixed by the capacity (blocks at or
  // beyond n_c are discarded when classified).
  const float* sc = a.scores + static_cast<int64_t>(b) * a.capacity;
  const int64_t chunk = (static_cast<int64_t>(a.capacity) + gridDim.x - 1) / gridDim.x;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * chunk;
  const int64_t cap_end = c0 + chunk < a.capacity ? c0 + chunk : a.capacity;
  uint32_t* cnt = a.cnt + b * kCntWords;
  int64_t n_c = vseq_tokens(a.n_tokens, b, a.T) / a.ratio;
  if (n_c > a.capacity) n_c = a.capacity;
  int32_t* out = a.topk + static_cast<int64_t>(b) * a.k;
  const int k = a.k;
  if (n_c <= k) {
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < n_c ? i : -1;
    return;
  }
  int32_t* above = a.above + static_cast<int64_t>(b) * k;
  uint64_t* cand = a.cand + static_cast<int64_t>(b) * a.capacity;

  uint32_t* hist2 = a.hist2 + static_cast<int64_t>(b) * kBins;
  // the first-level threshold bin T1 (the bin holding the k-th largest key)
  // from the scoring kernel's full histogram, found by every CTA
  {
    const uint32_t* gh = a.hist1 + static_cast<int64_t>(b) * kBins;
    constexpr int per = kBins / kSelThreads;
    uint32_t v[per];
#pragma unroll
    for (int u = 0; u < per; ++u) v[u] = __ldcg(gh + threadIdx.x + u * kSelThreads);
#pragma unroll
    for (int u = 0; u < per; ++u) h[threadIdx.x + u * kSelThreads] = v[u];
  }
  __syncthreads();
  uint32_t n_gt1;
  const uint32_t T1 = static_cast<uint32_t>(block_suffix_select<kSelThreads>(h, static_cast<uint32_t>(k), &n_gt1, scratch));
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int64_t c1 = cap_end < n_c ? cap_end : n_c;
  for (int64_t base = c0; base < c1; base += kScanItems * blockDim.x) {
    uint32_t key[kScanItems];
#pragma unroll
    for (int u = 0; u < kScanItems; ++u) {
      const int64_t s = base + threadIdx.x + u * blockDim.x;
      key[u] = s < c1 ? score_key(__ldg(sc + s)) : 0u;
    }
    uint32_t mine = 0;   // packed counts: above T1 (low 16 bits), in T1 (high 16 bits)
#pragma unroll
    for (int u = 0; u < kScanItems; ++u) {
      const int64_t s = base + threadIdx.x + u * blockDim.x;
      const bool in = s < c1;
      const uint32_t bin = key[u] >> 20;
      mine += (in && bin > T1) ? 1u : 0u;
      mine += (in && bin == T1) ? (1u << 16) : 0u;
      warp_hist_add(h, (key[u] >> 8) & 0xFFF, in && bin == T1);
    }
    uint32_t tot;
    uint32_t pre = block_excl_scan_packed(mine, &tot, scratch);
    if (threadIdx.x == 0) {
      s_base[0] = (tot & 0xFFFFu) ? atomicAdd(&cnt[0], tot & 0xFFFFu) : 0u;
      s_base[1] = (tot >> 16) ? atomicAdd(&cnt[1], tot >> 16) : 0u;
    }
    __syncthreads();
    uint32_t pg = s_base[0] + (pre & 0xFFFFu), pe = s_base[1] + (pre >> 16);
#pragma unroll
    for (int u = 0; u < kScanItems; ++u) {
      const int64_t s = base + threadIdx.x + u * blockDim.x;
      const bool in = s < c1;
      const uint32_t bin = key[u] >> 20;
      if (in && bin > T1) {
        if (pg < static_cast<uint32_t>(k)) above[pg] = static_cast<int32_t>(s);
        ++pg;
      } else if (in && bin == T1) {
        if (pe < static_cast<uint32_t>(a.capacity))
          cand[pe] = (static_cast<uint64_t>(key[u]) << 32) | static_cast<uint32_t>(s);
        ++pe;
      }
    }
    __syncthreads();
  }
  for (int i = threadIdx.x; i < kBins; i += blockDim.x)
    if (h[i]) atomicAdd(&hist2[i], h[i]);
  // the CTA's appends and histogram atomics precede its completion count (the
  // fence after the barrier is cumulative over the CTA's writes)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&cnt[2], 1u) == gridDim.x - 1;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;

  // ---- the last CTA of sequence b resolves the boundary
  uint32_t n_above = __ldcg(&cnt[0]);
  uint32_t n_cand = __ldcg(&cnt[1]);
  if (n_above > static_cast<uint32_t>(k)) n_above = k;                      // only on inconsistent input
  if (n_cand > static_cast<uint32_t>(a.capacity)) n_cand = a.capacity;
  const uint32_t need1 = static_cast<uint32_t>(k) - n_above;                 // taken from cand
  if (n_cand <= static_cast<uint32_t>(kRegCand * kSelThreads)) {
    resolve_in_registers(k, n_c, n_above, n_cand, need1, hist2, above, cand, out, h, fin, h8, scratch, dyn,
                         &s_nfin, &s_d, &s_rem);
    return;
  }
  load_to_smem(h, hist2, kBins);
  load_to_smem(fin, above, n_above);
  if (threadIdx.x == 0) s_nfin = n_above;
  uint64_t* cache = dyn;
  const bool cached = n_cand <= static_cast<uint32_t>(kCandCache);
  if (cached) load_to_smem(cache, static_cast<const uint64_t*>(cand), n_cand);
  const uint64_t* cl = cached ? cache : cand;
  __syncthreads();
  uint32_t n_gt2 = 0;
  const uint32_t T2 = need1 ? static_cast<uint32_t>(block_suffix_select<kSelThreads>(h, need1, &n_gt2, scratch)) : 0xFFFFu;
  const uint32_t need2 = need1 - n_gt2;                                      // taken among the keys of bin (T1, T2)
  const uint32_t n_eq2 = T2 < static_cast<uint32_t>(kBins) ? h[T2] : 0u;

  // Within bin (T1, T2) the need2 best by (low 8 key bits desc, index asc):
  // every key with low8 > d8, and the r8 lowest indices with low8 == d8, i.e.
  // those <= thr (a radix select over 12-bit index digits, lowest first).
  uint32_t d8 = 0, thr = 0;
  if (need2 > 0 && need2 < n_eq2) {
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
    __syncthreads();
    for (uint32_t i0 = 0; i0 < n_cand; i0 += blockDim.x) {
      const uint32_t i = i0 + threadIdx.x;
      const uint64_t v = i < n_cand ? cl[i] : 0ull;
      const uint32_t key = static_cast<uint32_t>(v >> 32);
      warp_hist_add(h, key & 0xFF, i < n_cand && ((key >> 8) & 0xFFF) == T2);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      s_d = 0;
      s_rem = 0;
    }
    __syncthreads();
    if (threadIdx.x < 32) warp_digit_select(h, need2, &s_d, &s_rem);
    __syncthreads();
    d8 = s_d;
    uint32_t r8 = need2 - s_rem;   // lowest indices to take among low8 == d8
    int nbits = 1;
    while (nbits < 31 && (static_cast<int64_t>(1) << nbits) < n_c) ++nbits;
    const int passes = (nbits + 11) / 12;
    uint32_t prefix = 0;
    for (int pass = 0; pass < passes; ++pass) {
      const int shift = 12 * (passes - 1 - pass);
      __syncthreads();
      for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
      __syncthreads();
      for (uint32_t i0 = 0; i0 < n_cand; i0 += blockDim.x) {
        const uint32_t i = i0 + threadIdx.x;
        const uint64_t v = i < n_cand ? cl[i] : 0ull;
        const uint32_t key = static_cast<uint32_t>(v >> 32), idx = static_cast<uint32_t>(v);
        const bool in = i < n_cand && ((key >> 8) & 0xFFF) == T2 && (key & 0xFF) == d8 &&
                        (pass == 0 || (idx >> (shift + 12)) == prefix);
        // reversed digit: the largest reversed bin with enough keys at or above it is the smallest digit
        warp_hist_add(h, (kBins - 1) - ((idx >> shift) & 0xFFF), in);
      }
      __syncthreads();
      uint32_t before;
      const uint32_t rd = static_cast<uint32_t>(block_suffix_select<kSelThreads>(h, r8, &before, scratch));
      prefix = (prefix << 12) | ((kBins - 1) - rd);
      r8 -= before;
    }
    thr = prefix;   // exactly the wanted number of indices with low8 == d8 are <= thr
  }
  __syncthreads();
  for (uint32_t i0 = 0; i0 < n_cand; i0 += blockDim.x) {
    const uint32_t i = i0 + threadIdx.x;
    const uint64_t v = i < n_cand ? cl[i] : 0ull;
    const uint32_t key = static_cast<uint32_t>(v >> 32), idx = static_cast<uint32_t>(v);
    const uint32_t b2 = (key >> 8) & 0xFFF;
    bool take = i < n_cand && need1 > 0 && b2 > T2;
    if (i < n_cand && b2 == T2 && need2 > 0)
      take = need2 >= n_eq2 || (key & 0xFF) > d8 || ((key & 0xFF) == d8 && idx <= thr);
    warp_append_i32(take, static_cast<int32_t>(idx), &s_nfin, fin, static_cast<uint32_t>(k));
  }
  __syncthreads();
  // the k blocks in ascending index order (padding -1 only on inconsistent input)
  const uint32_t nf = s_nfin < static_cast<uint32_t>(k) ? s_nfin : static_cast<uint32_t>(k);
  int P = 1;
  while (P < k) P <<= 1;
  for (int i = threadIdx.x + static_cast<int>(nf); i < P; i += blockDim.x) fin[i] = 0x7FFFFFFF;
  __syncthreads();
  block_sort_asc(fin, P);
  for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < static_cast<int>(nf) ? fin[i] : -1;
}

int launch_topk_select(const IndexArgs& a, int sel_ctas, cudaStream_t st) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTopkDynSmem);
  });
  return launch_pdl(topk_select_kernel, dim3(sel_ctas, a.B), dim3(kSelThreads), kTopkDynSmem, st, a);
}

}  // namespace dsv4
