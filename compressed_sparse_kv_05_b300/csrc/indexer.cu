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
#include "tc_ptx.cuh"

namespace dsv4 {

// grid (B * N), block Di/16: quantise one query head to FP4 (the same rule as the
// keys) into the operand layout of the scoring MMA; padding heads (h >= Hi) get
// zero codes and zero scales.
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

// ------------------------------------------------------------------------------ cluster top-k
//
// The same selection (the k largest score keys, ties to the lower index, in
// ascending index order) by one thread-block cluster of up to 16 CTAs per
// sequence, without global atomics or a resolving CTA. CTA r of the cluster
// copies scores [r S, (r + 1) S) of the sequence into shared memory (one bulk
// copy) while it finds T1, the top-12-bit bin holding the k-th largest key,
// in the scoring kernel's histogram; it then keeps the keys at or above bin
// T1 (a few hundred in a sequence, typically) as a list of (key, position).
// The boundary key is found digit by digit from histograms of the next 12 and
// the low 8 bits that every CTA adds into every CTA's shared memory
// (distributed shared memory), so that each finds the digit itself; a level
// is skipped when its boundary bin is taken whole. Every CTA then counts its keys above the boundary and equal to
// it; from the cluster's counts (ascending index ranges) it knows how many of
// its boundary keys it takes (the lowest indices) and where its selection
// starts in the output, and writes its selection in index order (each
// selected key's rank by counting the CTA's smaller positions). A CTA whose
// list would overflow works on all of its keys instead (positions in index
// order from warp ballots and block-wide prefix sums).

namespace {

constexpr int kClThreads = 512;
constexpr int kClWarps = kClThreads / 32;
constexpr int kClMaxCtas = 16;
constexpr int kClList = kBins / 2;   // list entries (uint2) in the first-level histogram's place
constexpr int kClRecv = 4096;        // keys of the boundary bin the first CTA receives (uint2)

DSV4_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
DSV4_DEV uint32_t cluster_ctas() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// address of shared variable p in the shared memory of cluster CTA `rank`
DSV4_DEV uint32_t peer_addr(const void* p, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(a), "r"(rank));
  return out;
}
DSV4_DEV void peer_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
DSV4_DEV void peer_store(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
DSV4_DEV uint32_t peer_fetch_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
DSV4_DEV void peer_store2(uint32_t addr, uint2 v) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}
// cluster-wide barrier (every thread of every CTA), split into its two halves
DSV4_DEV void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
DSV4_DEV void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
DSV4_DEV void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

// Add 1 to bin `bin` of the histogram `hist` (shared memory) of every CTA of
// the cluster, for every lane with `active`: per distinct bin of the warp,
// lanes 0..cs-1 each add the bin's count into one CTA. All 32 lanes call it.
DSV4_DEV void warp_hist_add_all(uint32_t* hist, uint32_t cs, uint32_t bin, bool active) {
  unsigned todo = __ballot_sync(0xffffffffu, active);
  const int lane = threadIdx.x & 31;
  const unsigned mine = __match_any_sync(0xffffffffu, active ? bin : 0xFFFFFFFFu);
  while (todo) {
    const int src = __ffs(todo) - 1;
    const unsigned grp = __shfl_sync(0xffffffffu, mine, src);   // the lanes sharing src's bin
    const uint32_t b = __shfl_sync(0xffffffffu, bin, src);
    if (lane < static_cast<int>(cs)) peer_add(peer_addr(hist + b, lane), static_cast<uint32_t>(__popc(grp & todo)));
    todo &= ~grp;
  }
}

// In-place exclusive prefix sum of n <= 4 * kClThreads words of shared memory.
DSV4_DEV void block_excl_scan_words(uint32_t* v, int n, uint32_t* scratch) {
  const int per = (n + kClThreads - 1) / kClThreads;
  const int i0 = threadIdx.x * per;
  uint32_t mine = 0;
  for (int i = 0; i < per; ++i)
    if (i0 + i < n) mine += v[i0 + i];
  uint32_t tot;
  uint32_t run = block_excl_scan_packed(mine, &tot, scratch);
  for (int i = 0; i < per; ++i)
    if (i0 + i < n) {
      const uint32_t c = v[i0 + i];
      v[i0 + i] = run;
      run += c;
    }
  __syncthreads();
}

template <int J>
constexpr size_t cluster_smem_bytes() {
  return static_cast<size_t>(J) * kClThreads * 4 + 2 * kBins * 4 + 2 * static_cast<size_t>(J / 4) * kClWarps * 4 +
         static_cast<size_t>(kClRecv) * 8;
}

}  // namespace

template <int J>
__global__ void __launch_bounds__(kClThreads, 1) topk_cluster_kernel(IndexArgs a) {
  constexpr int G = J / 4;                                 // groups of 4 * 512 scores
  extern __shared__ __align__(16) uint32_t dsm[];
  float* sv = reinterpret_cast<float*>(dsm);               // [G][512][4]: the CTA's scores; list mode: scratch
  uint32_t* h1 = dsm + J * kClThreads;                     // first-level histogram, then the candidate list
  uint2* list = reinterpret_cast<uint2*>(h1);              // (key, position) of the keys >= bin T1
  uint32_t* h2 = h1 + kBins;                               // the cluster's next-12-bit histogram
  uint32_t* pos_a = h2 + kBins;                            // full mode: per (group, warp) counts, then prefixes
  uint32_t* pos_b = pos_a + G * kClWarps;
  uint2* recv = reinterpret_cast<uint2*>(pos_b + G * kClWarps);   // first CTA: the cluster's keys of bin T1
  __shared__ uint32_t h8[256];                             // the cluster's low-8-bit histogram
  __shared__ uint32_t scratch[kClWarps + 2];
  __shared__ uint32_t all_cnt[2 * kClMaxCtas];             // every CTA's keys above / at the boundary
  __shared__ uint32_t s_d, s_above, s_list, s_nsel, s_neq;
  __shared__ uint32_t s_recv, s_ovf, s_slot;               // first CTA: keys received, overflow
  __shared__ uint32_t above_cnt[kClMaxCtas], sel_cnt[kClMaxCtas];
  __shared__ uint32_t res[5];                              // from the first CTA: overflow, Kx, tie, pthr, base
  __shared__ uint64_t landed[G];                           // bulk copy of group g
  __shared__ int abort_flag;
  pdl_trigger();
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  for (int i = t; i < kBins; i += kClThreads) h2[i] = 0;
  if (t < 256) h8[t] = 0;
  if (t == 0) {
    for (int g = 0; g < G; ++g) tc::mbar_init(&landed[g], 1);
    abort_flag = 0;
    s_list = 0;
    s_recv = 0;
    s_ovf = 0;
    s_nsel = 0;
    s_neq = 0;
    tc::fence_mbar_init();
  }
  cluster_arrive();   // phase 0: every CTA's histograms are zeroed before anyone adds into them
  pdl_wait();
  const int b = blockIdx.y;
  const uint32_t r = cluster_rank(), cs = cluster_ctas();
  int64_t n_c = vseq_tokens(a.n_tokens, b, a.T) / a.ratio;
  if (n_c > a.capacity) n_c = a.capacity;
  const int k = a.k;
  int32_t* out = a.topk + static_cast<int64_t>(b) * k;
  if (n_c <= k) {   // uniform across the cluster
    if (r == 0)
      for (int i = t; i < k; i += kClThreads) out[i] = i < n_c ? i : -1;
    cluster_wait();
    return;
  }
  // CTA r: scores [lo, lo + nl), S a multiple of 4 so that a slice starts on
  // a 16-byte boundary whenever a sequence's row does (the host keeps S <= 512 J)
  const int64_t S = (((n_c + cs - 1) / cs) + 3) & ~int64_t(3);
  const int64_t lo = static_cast<int64_t>(r) * S;
  const int nl = static_cast<int>(n_c - lo < S ? (n_c - lo > 0 ? n_c - lo : 0) : S);
  const float* sc = a.scores + static_cast<int64_t>(b) * a.capacity + lo;
  // the slice into shared memory: one bulk copy per group of its whole 16-byte
  // granules when aligned, the rest (or everything) by plain loads
  const bool bulk = (reinterpret_cast<uintptr_t>(sc) & 15) == 0;
  const int nbulk = bulk ? (nl & ~3) : 0;
  __syncthreads();
  if (t == 0)
    for (int g = 0; g < G && g * 2048 < nbulk; ++g) {
      const int n = nbulk - g * 2048 < 2048 ? nbulk - g * 2048 : 2048;
      tc::mbar_arrive_expect_tx(&landed[g], static_cast<uint32_t>(n) * 4u);
      tc::bulk_load(sv + g * 2048, sc + g * 2048, static_cast<uint32_t>(n) * 4u, &landed[g]);
    }
  for (int e = nbulk + t; e < nl; e += kClThreads) sv[e] = __ldcg(sc + e);
  {
    const uint32_t* gh = a.hist1 + static_cast<int64_t>(b) * kBins;
    constexpr int per = kBins / kClThreads;
    uint32_t v[per];
#pragma unroll
    for (int u = 0; u < per; ++u) v[u] = __ldcg(gh + t + u * kClThreads);
#pragma unroll
    for (int u = 0; u < per; ++u) h1[t + u * kClThreads] = v[u];
  }
  __syncthreads();
  uint32_t n_gt1;
  const uint32_t T1 = static_cast<uint32_t>(block_suffix_select<kClThreads>(h1, static_cast<uint32_t>(k), &n_gt1, scratch));
  const uint32_t need1 = static_cast<uint32_t>(k) - n_gt1;
  const uint32_t cnt1 = h1[T1];
  __syncthreads();   // h1 is read; it becomes the candidate list
  // Keys at or above bin T1 into the list (one shared-memory slot each, in no
  // particular order). A float test that admits every such score (and NaN)
  // comes first; the key decides.
  const uint32_t kmin = T1 << 20;
  float fthr;
  {
    const uint32_t u = (kmin & 0x80000000u) ? (kmin & 0x7FFFFFFFu) : ~kmin;
    fthr = __uint_as_float(u);
    if (fthr != fthr) fthr = (kmin & 0x80000000u) ? INFINITY : -INFINITY;
  }
  for (int g = 0; g < G; ++g) {
    if (g * 2048 < nbulk && !tc::mbar_wait(&landed[g], 0, &abort_flag)) atomicOr(a.status, DSV4_STATUS_TIMEOUT);
    const int p = g * 2048 + 4 * t;
    if (p >= nl) continue;
    float4 f;
    if (p + 3 < nl) {
      f = *reinterpret_cast<const float4*>(sv + p);
    } else {
      f.x = sv[p];
      f.y = p + 1 < nl ? sv[p + 1] : -INFINITY;
      f.z = p + 2 < nl ? sv[p + 2] : -INFINITY;
      f.w = -INFINITY;
    }
    if (!(f.x < fthr) || !(f.y < fthr) || !(f.z < fthr) || !(f.w < fthr)) {
      const float fs[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t key = score_key(fs[i]);
        if (p + i < nl && key >= kmin) {
          const uint32_t slot = atomicAdd(&s_list, 1u);
          if (slot < static_cast<uint32_t>(kClList)) list[slot] = make_uint2(key, static_cast<uint32_t>(p + i));
        }
      }
    }
  }
  __syncthreads();
  const uint32_t L = s_list;
  const bool full = L > static_cast<uint32_t>(kClList);   // uniform within the CTA
  cluster_wait();

  // ---- Usual case: the first CTA resolves the boundary among the keys of bin
  // T1 (cnt1 of them), which every CTA sends it as (key, r << 16 | position),
  // with its count of keys above bin T1; it returns to each CTA the boundary
  // key, whether it ties, the CTA's last boundary position taken and where its
  // selection starts.
  {
    const uint32_t leader = 0;
    uint32_t n_in = 0, n_up = 0;   // this thread's list entries in bin T1 / above it
    if (!full)
      for (uint32_t i = t; i < L; i += kClThreads) {
        const uint32_t bin = list[i].x >> 20;
        n_in += bin == T1 ? 1u : 0u;
        n_up += bin > T1 ? 1u : 0u;
      }
    uint32_t tot;
    const uint32_t off = block_excl_scan_packed(n_in | (n_up << 16), &tot, scratch);
    if (t == 0) {
      if (full) {
        peer_store(peer_addr(&s_ovf, leader), 1u);
      } else {
        s_slot = (tot & 0xFFFFu) ? peer_fetch_add(peer_addr(&s_recv, leader), tot & 0xFFFFu) : 0u;
        peer_store(peer_addr(&above_cnt[r], leader), tot >> 16);
      }
    }
    __syncthreads();
    if (!full && n_in) {
      uint32_t slot = s_slot + (off & 0xFFFFu);
      for (uint32_t i = t; i < L; i += kClThreads) {
        const uint2 en = list[i];
        if ((en.x >> 20) == T1) {
          if (slot < static_cast<uint32_t>(kClRecv)) peer_store2(peer_addr(&recv[slot], leader), make_uint2(en.x, (r << 16) | en.y));
          ++slot;
        }
      }
    }
  }
  cluster_sync();   // phase 1: the first CTA holds the cluster's keys of bin T1
  if (r == 0) {
    const uint32_t R = s_recv;
    const bool ovf = s_ovf != 0 || R > static_cast<uint32_t>(kClRecv) || R != cnt1;
    uint32_t Kr = kmin, tie_r = 0, qthr = 0;
    if (!ovf) {
      if (t < kClMaxCtas) sel_cnt[t] = 0;
      if (need1 < cnt1) {
        for (uint32_t i = t; i < R; i += kClThreads) atomicAdd(&h2[(recv[i].x >> 8) & 0xFFFu], 1u);
        __syncthreads();
        uint32_t n_gt2;
        const uint32_t T2 = static_cast<uint32_t>(block_suffix_select<kClThreads>(h2, need1, &n_gt2, scratch));
        const uint32_t need2 = need1 - n_gt2, cnt2 = h2[T2];
        const uint32_t p24 = (T1 << 12) | T2;
        Kr = p24 << 8;
        if (need2 < cnt2) {
          for (uint32_t i = t; i < R; i += kClThreads)
            if ((recv[i].x >> 8) == p24) atomicAdd(&h8[recv[i].x & 0xFFu], 1u);
          __syncthreads();
          if (w == 0) warp_digit_select(h8, need2, &s_d, &s_above);
          __syncthreads();
          const uint32_t d8 = s_d, need3 = need2 - s_above, cnt3 = h8[d8];
          Kr = (p24 << 8) | d8;
          if (need3 < cnt3) {
            // the need3 lowest cluster positions q among the keys == Kr: a
            // radix select over q's 20 bits (digits 8, 8, 4), smallest first
            tie_r = 1;
            uint32_t rneed = need3, prefix = 0;
            const int shifts[3] = {12, 4, 0};
            const int widths[3] = {8, 8, 4};
            for (int ps = 0; ps < 3; ++ps) {
              __syncthreads();
              if (t < 256) h8[t] = 0;
              __syncthreads();
              const int sh = shifts[ps];
              for (uint32_t i = t; i < R; i += kClThreads) {
                const uint2 en = recv[i];
                if (en.x == Kr && (ps == 0 || (en.y >> (sh + widths[ps])) == prefix))
                  atomicAdd(&h8[255u - ((en.y >> sh) & ((1u << widths[ps]) - 1u))], 1u);
              }
              __syncthreads();
              if (w == 0) warp_digit_select(h8, rneed, &s_d, &s_above);
              __syncthreads();
              prefix = (prefix << widths[ps]) | (255u - s_d);
              rneed -= s_above;
            }
            qthr = prefix;   // exactly need3 keys == Kr have q <= qthr
          }
        }
      }
      __syncthreads();
      for (uint32_t i = t; i < R; i += kClThreads) {
        const uint2 en = recv[i];
        const bool sel = en.x > Kr || (en.x == Kr && (!tie_r || en.y <= qthr));
        if (sel) atomicAdd(&sel_cnt[en.y >> 16], 1u);
      }
      __syncthreads();
    }
    if (t < static_cast<int>(cs)) {
      uint32_t base_t = 0;
      for (int q = 0; q < t; ++q) base_t += above_cnt[q] + sel_cnt[q];
      int32_t pthr = -1;
      if (tie_r) {
        const int qr = static_cast<int>(qthr >> 16);
        pthr = t < qr ? 0xFFFF : t == qr ? static_cast<int32_t>(qthr & 0xFFFFu) : -1;
      }
      peer_store(peer_addr(&res[0], t), ovf ? 1u : 0u);
      peer_store(peer_addr(&res[1], t), Kr);
      peer_store(peer_addr(&res[2], t), tie_r);
      peer_store(peer_addr(&res[3], t), static_cast<uint32_t>(pthr));
      peer_store(peer_addr(&res[4], t), base_t);
    }
  }
  cluster_sync();   // phase 2: every CTA holds the first CTA's answer
  if (res[0] == 0) {
    // this CTA's selection (its list: no CTA is in full mode here), each
    // entry's rank among them by counting smaller positions
    const uint32_t Kr = res[1], base_r = res[4];
    const bool tie_r = res[2] != 0;
    const int32_t pthr = static_cast<int32_t>(res[3]);
    uint32_t* selp = reinterpret_cast<uint32_t*>(sv);   // free: every key of interest is in the list
    for (uint32_t i0 = 0; i0 < L; i0 += kClThreads) {
      const uint32_t i = i0 + t;
      bool sel = false;
      uint32_t p = 0;
      if (i < L) {
        const uint2 en = list[i];
        p = en.y;
        sel = en.x > Kr || (en.x == Kr && (!tie_r || static_cast<int32_t>(p) <= pthr));
      }
      warp_append_i32(sel, static_cast<int32_t>(p), &s_nsel, reinterpret_cast<int32_t*>(selp), static_cast<uint32_t>(k));
    }
    __syncthreads();
    const uint32_t ns = s_nsel < static_cast<uint32_t>(k) ? s_nsel : static_cast<uint32_t>(k);
    for (uint32_t i = t; i < ns; i += kClThreads) {
      const uint32_t p = selp[i];
      uint32_t rank = 0;
      for (uint32_t q = 0; q < ns; ++q) rank += selp[q] < p ? 1u : 0u;
      if (base_r + rank < static_cast<uint32_t>(k)) out[base_r + rank] = static_cast<int32_t>(lo + p);
    }
    return;
  }
  // ---- Otherwise (a CTA with too many keys at or above bin T1, or too many
  // keys in bin T1 for the first CTA, which then left its histograms at zero):
  // digit by digit across the cluster.

  // The boundary: with tie == false every key >= Kx is taken; with tie ==
  // true every key > Kx and the `need` lowest-index keys == Kx. Every key not
  // in a CTA's list is below bin T1, so below Kx.
  uint32_t Kx = kmin, need = 0;
  bool tie = false;
  // calls f(key, valid) for every key of the CTA at or above bin T1 (the list,
  // or all keys), with whole warps
  auto for_each_candidate = [&](auto&& f) {
    if (!full) {
      for (uint32_t i0 = 0; i0 < L; i0 += kClThreads) {
        const uint32_t i = i0 + t;
        const uint2 e = i < L ? list[i] : make_uint2(0u, 0u);
        f(e.x, i < L);
      }
    } else {
      for (int g = 0; g < G; ++g) {
        const int p = g * 2048 + 4 * t;
#pragma unroll
        for (int i = 0; i < 4; ++i) f(p + i < nl ? score_key(sv[p + i]) : 0u, p + i < nl);
      }
    }
  };
  // adds 1 at bin(key) of histogram `hist` in every CTA for every key of this
  // CTA at or above bin T1 with in(key): list mode, one remote add per
  // (entry, CTA) pair spread over the threads; else warp-aggregated
  auto add_all = [&](uint32_t* hist, auto&& in, auto&& bin) {
    if (!full) {
      for (uint32_t i = t; i < L * cs; i += kClThreads) {
        const uint32_t key = list[i / cs].x;
        if (in(key)) peer_add(peer_addr(hist + bin(key), i % cs), 1u);
      }
    } else {
      for_each_candidate([&](uint32_t key, bool v) { warp_hist_add_all(hist, cs, bin(key), v && in(key)); });
    }
  };
  if (need1 < cnt1) {
    add_all(h2, [&](uint32_t key) { return (key >> 20) == T1; }, [](uint32_t key) { return (key >> 8) & 0xFFFu; });
    cluster_sync();   // phase 1: every CTA holds the cluster's next-12-bit histogram
    uint32_t n_gt2;
    const uint32_t T2 = static_cast<uint32_t>(block_suffix_select<kClThreads>(h2, need1, &n_gt2, scratch));
    const uint32_t need2 = need1 - n_gt2, cnt2 = h2[T2];
    const uint32_t p24 = (T1 << 12) | T2;
    Kx = p24 << 8;
    if (need2 < cnt2) {
      add_all(h8, [&](uint32_t key) { return (key >> 8) == p24; }, [](uint32_t key) { return key & 0xFFu; });
      cluster_sync();   // phase 2: every CTA holds the cluster's low-8-bit histogram
      if (w == 0) warp_digit_select(h8, need2, &s_d, &s_above);
      __syncthreads();
      const uint32_t d8 = s_d, need3 = need2 - s_above, cnt3 = h8[d8];
      Kx = (p24 << 8) | d8;
      if (need3 < cnt3) {
        tie = true;
        need = need3;
      }
    }
  }

  // this CTA's keys above the boundary (>= Kx without a tie) and at it
  uint32_t g = 0, e = 0;
  for_each_candidate([&](uint32_t key, bool v) {
    g += (v && (tie ? key > Kx : key >= Kx)) ? 1u : 0u;
    e += (v && tie && key == Kx) ? 1u : 0u;
  });
  {
    uint32_t ge;   // both counts in one sum (each below 2^16: a CTA holds at most 512 J keys)
    block_excl_scan_packed(g | (e << 16), &ge, scratch);
    g = ge & 0xFFFFu;
    e = ge >> 16;
  }
  if (t < static_cast<int>(cs)) {
    peer_store(peer_addr(&all_cnt[2 * r], t), g);
    peer_store(peer_addr(&all_cnt[2 * r + 1], t), e);
  }
  cluster_sync();   // phase 3: every CTA holds every CTA's counts; no shared memory is touched remotely after this
  // the boundary keys this CTA takes and where its selection starts
  uint32_t base = 0, eq_before = 0, take = 0;
  for (uint32_t q = 0; q < cs; ++q) {
    const uint32_t cq = all_cnt[2 * q + 1];
    const uint32_t tq = tie ? (need > eq_before ? (need - eq_before < cq ? need - eq_before : cq) : 0u) : 0u;
    if (q < r) base += all_cnt[2 * q] + tq;
    if (q == r) take = tq;
    eq_before += cq;
  }
  const bool split = tie && take > 0 && take < e;   // uniform within the CTA
  const unsigned below = (1u << lane) - 1u;

  if (!full) {
    // positions of the boundary keys (split only), then of the selected keys,
    // gathered in list order; each one's rank is the count of smaller positions
    uint32_t* eqp = h2;                               // free again: no CTA adds into it after phase 1
    uint32_t* selp = reinterpret_cast<uint32_t*>(sv);  // free: every key of interest is in the list
    if (split) {
      for (uint32_t i0 = 0; i0 < L; i0 += kClThreads) {
        const uint32_t i = i0 + t;
        const bool at_b = i < L && list[i].x == Kx;
        warp_append_i32(at_b, static_cast<int32_t>(i < L ? list[i].y : 0u), &s_neq, reinterpret_cast<int32_t*>(eqp),
                        static_cast<uint32_t>(kBins));
      }
      __syncthreads();
    }
    for (uint32_t i0 = 0; i0 < L; i0 += kClThreads) {
      const uint32_t i = i0 + t;
      bool sel = false;
      uint32_t p = 0;
      if (i < L) {
        const uint2 en = list[i];
        p = en.y;
        sel = tie ? en.x > Kx : en.x >= Kx;
        if (tie && en.x == Kx) {
          if (!split) {
            sel = take > 0;
          } else {
            uint32_t rank = 0;
            for (uint32_t q = 0; q < e; ++q) rank += eqp[q] < p ? 1u : 0u;
            sel = rank < take;
          }
        }
      }
      warp_append_i32(sel, static_cast<int32_t>(p), &s_nsel, reinterpret_cast<int32_t*>(selp), static_cast<uint32_t>(k));
    }
    __syncthreads();
    const uint32_t ns = s_nsel < static_cast<uint32_t>(k) ? s_nsel : static_cast<uint32_t>(k);
    for (uint32_t i = t; i < ns; i += kClThreads) {
      const uint32_t p = selp[i];
      uint32_t rank = 0;
      for (uint32_t q = 0; q < ns; ++q) rank += selp[q] < p ? 1u : 0u;
      if (base + rank < static_cast<uint32_t>(k)) out[base + rank] = static_cast<int32_t>(lo + p);
    }
  } else {
    // every key of the CTA, in index order: group g, warp w covers positions
    // g 2048 + 128 w ..., lane by lane, 4 per lane; a (group, warp) count from
    // four ballots, block-wide prefix sums over (group, warp)
    auto key_at = [&](int p) { return p < nl ? score_key(sv[p]) : 0u; };
    if (split) {
      for (int gg = 0; gg < G; ++gg) {
        const int p = gg * 2048 + 4 * t;
        uint32_t c = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) c += __popc(__ballot_sync(0xffffffffu, p + i < nl && key_at(p + i) == Kx));
        if (lane == 0) pos_a[gg * kClWarps + w] = c;
      }
      __syncthreads();
      block_excl_scan_words(pos_a, G * kClWarps, scratch);
    }
    // selection flags of this thread's 4 keys of group gg, and the count of
    // selected keys before them within the (group, warp)
    auto select4 = [&](int gg, bool* sel, uint32_t* before) {
      const int p = gg * 2048 + 4 * t;
      bool at[4];
      uint32_t eq_rank = split ? pos_a[gg * kClWarps + w] : 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t key = key_at(p + i);
        const bool v = p + i < nl;
        sel[i] = v && (tie ? key > Kx : key >= Kx);
        at[i] = v && tie && key == Kx;
      }
      if (split) {
        uint32_t lower = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) lower += __popc(__ballot_sync(0xffffffffu, at[i]) & below);
        eq_rank += lower;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sel[i] |= at[i] && eq_rank < take;
          eq_rank += at[i] ? 1u : 0u;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) sel[i] |= at[i] && take > 0;
      }
      uint32_t lower = 0, cnt = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const unsigned m = __ballot_sync(0xffffffffu, sel[i]);
        lower += __popc(m & below);
        cnt += __popc(m);
      }
      *before = lower;
      return cnt;
    };
    for (int gg = 0; gg < G; ++gg) {
      bool sel[4];
      uint32_t before;
      const uint32_t c = select4(gg, sel, &before);
      if (lane == 0) pos_b[gg * kClWarps + w] = c;
    }
    __syncthreads();
    block_excl_scan_words(pos_b, G * kClWarps, scratch);
    for (int gg = 0; gg < G; ++gg) {
      bool sel[4];
      uint32_t before;
      select4(gg, sel, &before);
      uint32_t pos = base + pos_b[gg * kClWarps + w] + before;
      const int p = gg * 2048 + 4 * t;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (sel[i]) {
          if (pos < static_cast<uint32_t>(k)) out[pos] = static_cast<int32_t>(lo + p + i);
          ++pos;
        }
    }
  }
}

namespace {
constexpr int kClJ[3] = {16, 36, 72};   // scores per thread of the instantiated cluster kernels

template <int J>
void cluster_setup() {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(topk_cluster_kernel<J>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(cluster_smem_bytes<J>()));
    cudaFuncSetAttribute(topk_cluster_kernel<J>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
}

template <int J>
cudaLaunchConfig_t cluster_config(int cs, int B, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, B);
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = cluster_smem_bytes<J>();
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cs;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// whether clusters of cs CTAs of topk_cluster_kernel<J> can be resident on this device
template <int J>
bool cluster_fits(int cs) {
  cluster_setup<J>();
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster_config<J>(cs, 1, nullptr, attr);
  cfg.attrs = attr + 1;   // the cluster shape alone
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, topk_cluster_kernel<J>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return n > 0;
}

bool cluster_fits_j(int J, int cs) {
  static int memo[3][5] = {};   // 0 unknown, 1 fits, 2 does not (per J, cs = 1 << i)
  int ji = J == kClJ[0] ? 0 : J == kClJ[1] ? 1 : 2, ci = 0;
  while ((1 << ci) < cs) ++ci;
  int& m = memo[ji][ci];
  if (!m) {
    const bool ok = ji == 0 ? cluster_fits<kClJ[0]>(cs) : ji == 1 ? cluster_fits<kClJ[1]>(cs) : cluster_fits<kClJ[2]>(cs);
    m = ok ? 1 : 2;
  }
  return m == 1;
}

template <int J>
int launch_topk_cluster(const IndexArgs& a, int cs, cudaStream_t st) {
  cluster_setup<J>();
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster_config<J>(cs, a.B, st, attr);
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel<J>, a) == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
}  // namespace

int topk_plan(int B, int capacity, int sms, int* cluster_ctas, int* per_thread) {
  for (int cs = kClMaxCtas; cs >= 1; cs >>= 1) {
    if (cs > 1 && B * cs > sms) continue;
    const int64_t per_cta = (((static_cast<int64_t>(capacity) + cs - 1) / cs) + 3) & ~int64_t(3);
    const int64_t need = (per_cta + kClThreads - 1) / kClThreads;
    for (int J : kClJ)
      if (need <= J && cluster_fits_j(J, cs)) {
        *cluster_ctas = cs;
        *per_thread = J;
        return 1;
      }
  }
  *cluster_ctas = 0;
  *per_thread = 0;
  return 0;
}

int launch_topk_select(const IndexArgs& a, int sel_ctas, int sms, cudaStream_t st) {
  int cs, J;
  if (topk_plan(a.B, a.capacity, sms, &cs, &J)) {
    if (J == kClJ[0]) return launch_topk_cluster<kClJ[0]>(a, cs, st);
    if (J == kClJ[1]) return launch_topk_cluster<kClJ[1]>(a, cs, st);
    return launch_topk_cluster<kClJ[2]>(a, cs, st);
  }
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTopkDynSmem);
  });
  return launch_pdl(topk_select_kernel, dim3(sel_ctas, a.B), dim3(kSelThreads), kTopkDynSmem, st, a);
}

}  // namespace dsv4
