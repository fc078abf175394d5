// Block-wide selection helpers for the top-k of the lightning indexer
// (vibecoco.ai, "DeepSeek V4 agent architecture", section
// "混合注意力：两种压缩，交替使用": the k highest-scoring compressed blocks are
// kept). Scores are compared through order-preserving unsigned keys
// (score_key in common.cuh); selection is a radix select over 12-bit digits.
#pragma once

#include "common.cuh"

namespace dsv4 {

constexpr int kBins = 4096;   // 12-bit digit histograms

// Barrier among threads [0, NT): the whole block (BAR = 0) or named barrier BAR.
template <int NT, int BAR>
DSV4_DEV void sync_threads_of() {
  if (BAR == 0) __syncthreads();
  else asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT) : "memory");
}

// Suffix search over a 4096-bin histogram h (shared memory) by NT threads,
// thread number tid in [0, NT) (threadIdx.x by default): the largest bin T
// with sum_{j >= T} h[j] >= need (need >= 1 and at most the histogram's
// total). Returns T in every thread and writes sum_{j > T} h[j] to *above.
// `scratch` is NT / 32 + 2 words of shared memory. BAR = 0: NT is the whole
// block; otherwise the named barrier BAR of those NT threads is used.
template <int NT, int BAR = 0>
DSV4_DEV int block_suffix_select(const uint32_t* h, uint32_t need, uint32_t* above, uint32_t* scratch,
                                 int tid = -1) {
  constexpr int per = kBins / NT;
  constexpr int nw = NT / 32;
  const int t = tid < 0 ? static_cast<int>(threadIdx.x) : tid, lane = t & 31, w = t >> 5;
  if (t == 0) {
    scratch[nw] = 0;
    scratch[nw + 1] = 0;
  }
  uint32_t mine = 0;
#pragma unroll
  for (int i = 0; i < per; ++i) mine += h[t * per + i];
  uint32_t suf = mine;   // sum over lanes >= lane of this warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += v;
  }
  if (lane == 0) scratch[w] = suf;
  sync_threads_of<NT, BAR>();
  uint32_t after = 0;
  for (int ww = w + 1; ww < nw; ++ww) after += scratch[ww];
  const uint32_t incl = suf + after;   // bins >= t * per
  const uint32_t excl = incl - mine;   // bins >= (t + 1) * per
  if (excl < need && incl >= need) {
    uint32_t acc = excl;
    for (int i = per - 1; i >= 0; --i) {
      const uint32_t c = h[t * per + i];
      if (acc + c >= need) {
        scratch[nw] = static_cast<uint32_t>(t * per + i);
        scratch[nw + 1] = acc;
        break;
      }
      acc += c;
    }
  }
  sync_threads_of<NT, BAR>();
  const int bin = static_cast<int>(scratch[nw]);
  *above = scratch[nw + 1];
  sync_threads_of<NT, BAR>();
  return bin;
}

// Add 1 to h[bin] for every lane with `active`, one atomic per distinct bin of
// the warp (lanes with equal bins are grouped), so that many equal keys do not
// serialise on one shared-memory word. All 32 lanes must call it.
DSV4_DEV void warp_hist_add(uint32_t* h, uint32_t bin, bool active) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (!act) return;
  const unsigned peers = __match_any_sync(0xffffffffu, active ? bin : 0xFFFFFFFFu) & act;
  const int lane = threadIdx.x & 31;
  if (active && (__ffs(peers) - 1) == lane) atomicAdd(&h[bin], static_cast<uint32_t>(__popc(peers)));
}

// Warp 0 of the block: the largest digit d of a 256-bin histogram h with
// sum_{j >= d} h[j] >= need, and sum_{j > d} h[j]. Other warps get nothing.
DSV4_DEV void warp_digit_select(const uint32_t* h, uint32_t need, uint32_t* digit, uint32_t* above) {
  const int lane = threadIdx.x & 31;
  uint32_t mine = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) mine += h[lane * 8 + i];
  uint32_t suf = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += v;
  }
  const uint32_t excl = suf - mine;
  if (excl < need && suf >= need) {
    uint32_t acc = excl;
    for (int i = 7; i >= 0; --i) {
      const uint32_t c = h[lane * 8 + i];
      if (acc + c >= need) {
        *digit = static_cast<uint32_t>(lane * 8 + i);
        *above = acc;
        break;
      }
      acc += c;
    }
  }
}

}  // namespace dsv4
