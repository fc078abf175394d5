// Lightning-indexer scores on the 5th-generation tensor cores (tcgen05,
// kind::mxf4nvf4 block-scaled FP4 MMA).
//
// vibecoco.ai, "DeepSeek V4 agent architecture", section
// "混合注意力：两种压缩，交替使用": the lightning indexer of CSA runs in FP4 and
// scores every compressed block with ReLU-scored multi-head dot products:
//   I_s = sum_h w_h * max(0, q_h . k_s).
// The contraction q_h . k_s is dense (all blocks x all indexer heads), so it
// runs as D[128 keys][N heads] = K_tile[128][Di] x Q[N][Di]^T per tile of 128
// compressed blocks, with the per-16 e4m3 scales of keys and query applied by
// the MMA itself (UE4M3 block scales). The epilogue applies ReLU and the head
// weights, writes one fp32 score per block and histograms the top 12 bits of
// the score keys for the top-k selection that follows (which finds the
// threshold bin in the full histogram).
//
// CTA roles (384 threads): warp 0 allocates tensor memory and streams key tiles
// with TMA into an S-stage ring; warp 1 issues tcgen05.cp (block scales) and
// the MMAs (one thread); warps 2-3 rearrange each tile's key scales in shared
// memory into the 32-row x 16-byte blocks that tcgen05.cp moves to tensor
// memory; warps 4-11 turn finished accumulators into scores, in two sets of
// four (one warp per 32-lane quarter of tensor memory) that take alternate
// tiles. The accumulator is double-buffered (one buffer per set) so the MMA
// of tile i+1 overlaps the epilogue of tile i.
//
// Scale block layout (one per 128 rows and K=64 step): row r's four scale bytes
// (one per 16 elements, the first in the lowest byte) form the 32-bit word at
// word index (r % 32) * 4 + r / 32.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "select.cuh"
#include "tc_ptx.cuh"

namespace dsv4 {

namespace {

constexpr int kTile = 128;     // compressed blocks per MMA tile (M)
constexpr int kThreads = 384;
constexpr int kEpiThreads = 256;   // warps 4-11
constexpr int kSfBlock = 512;  // bytes of one scale block (128 rows x 4 scales)

template <int ROWB>
struct TcCfg {
  static constexpr int KSTEPS = ROWB / 32;                   // K = 64 e2m1 values = 32 bytes per MMA
  static constexpr int STAGES = ROWB <= 64 ? 8 : 6;
  static constexpr int STAGE_BYTES = kTile * ROWB;
  static constexpr int SF_BYTES = KSTEPS * kSfBlock;          // one tile's key scales
  static constexpr uint32_t SWIZZLE = ROWB == 32 ? tc::kSwizzle32B : ROWB == 64 ? tc::kSwizzle64B : tc::kSwizzle128B;
  static constexpr int SF_COLS = 4 * KSTEPS;                  // tensor-memory columns of one tile's scales
};

struct SmemTail {
  uint64_t full[8], empty[8], sf_full[8], acc_full[2], acc_empty[2], q_full, qsf_full, drain;
  uint32_t taddr;
  int abort;
  uint32_t hist[kBins];  // histogram of score-key bits 31..20 of this CTA's blocks
};

// named barrier among the eight epilogue warps
DSV4_DEV void epilogue_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

}  // namespace

template <int ROWB>
__global__ void __launch_bounds__(kThreads, 2)
    index_scores_tc_kernel(const __grid_constant__ CUtensorMap keys, const __grid_constant__ CUtensorMap qmap,
                           IndexTcArgs a) {
  using C = TcCfg<ROWB>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;                                           // S x 128 x ROWB key codes
  unsigned char* qbuf = stages + C::STAGES * C::STAGE_BYTES;              // N x ROWB query codes
  unsigned char* sfbuf = qbuf + ((a.N * ROWB + 1023) & ~1023);           // S x SF_BYTES key scale blocks
  unsigned char* qsf = sfbuf + C::STAGES * C::SF_BYTES;                   // query scale blocks (N <= 128 rows)
  SmemTail* t = reinterpret_cast<SmemTail*>(qsf + C::SF_BYTES);
  float* wsm = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(t + 1) + 15) & ~uintptr_t(15));   // head weights
  pdl_trigger();
  if (threadIdx.x == 0) {
    tc::prefetch_tensormap(&keys);
    tc::prefetch_tensormap(&qmap);
  }
  if (threadIdx.x == 32 || threadIdx.x == 64) {
    // While the previous kernel finishes (the memory system is otherwise idle
    // then), this CTA's first ring's worth of key tiles is pulled into L2: a
    // hint, with the tile range of a full cache (the real range needs
    // n_tokens, read after the wait). Keys are only ever appended, and L2 is
    // coherent with the append's writes.
    const int tiles_c = static_cast<int>((static_cast<int64_t>(a.capacity) + kTile - 1) / kTile);
    const int per_c = (tiles_c + a.ctas_per_seq - 1) / a.ctas_per_seq;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * per_c * kTile;
    if (r0 < a.capacity) {
      const int64_t want = static_cast<int64_t>(C::STAGES) * kTile;
      const int64_t n = a.capacity - r0 < want ? a.capacity - r0 : want;
      const int64_t row = static_cast<int64_t>(blockIdx.y / a.T) * a.capacity + r0;
      // a sequence's slice of the scale plane starts on a 16-byte boundary only
      // when capacity * Di / 16 is a multiple of 16: the range helper trims it
      if (threadIdx.x == 32) tc::prefetch_l2_range(a.idx_codes + row * ROWB, n * ROWB);
      else tc::prefetch_l2_range(a.idx_scales + row * (ROWB / 8), n * (ROWB / 8));
    }
  }
  // head weights: the caller's input, which no kernel of this library writes
  // (heads beyond Hi weigh zero)
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) wsm[i] = i < a.Hi ? a.w[static_cast<int64_t>(blockIdx.y) * a.Hi + i] : 0.f;
  pdl_wait();

  const int b = blockIdx.y;              // virtual sequence (query)
  const int64_t bs = b / a.T;            // whose keys it scores
  int64_t n_c = vseq_tokens(a.n_tokens, b, a.T) / a.ratio;
  if (n_c > a.capacity) n_c = a.capacity;
  const int tiles = static_cast<int>((n_c + kTile - 1) / kTile);
  const int per = (tiles + a.ctas_per_seq - 1) / a.ctas_per_seq;
  const int t0 = blockIdx.x * per;
  const int t1 = t0 + per < tiles ? t0 + per : tiles;
  if (t0 >= t1) return;                                    // uniform across the CTA
  const int ntile = t1 - t0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const int nblk = ROWB / 8;                               // Di/16 scale bytes per row
  const uint32_t ncols = a.tmem_cols;
  const uint32_t acc_col0 = 0, sfa_col0 = 2 * N, sfb_col = 2 * N + 2 * C::SF_COLS;
  volatile int* abort = &t->abort;

  if (warp == 0) tc::tmem_alloc(&t->taddr, ncols);
  if (threadIdx.x == 32) {
    for (int i = 0; i < C::STAGES; ++i) {
      tc::mbar_init(&t->full[i], 1);
      tc::mbar_init(&t->empty[i], 1);
      tc::mbar_init(&t->sf_full[i], 2);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&t->acc_full[i], 1);
      tc::mbar_init(&t->acc_empty[i], 4);
    }
    tc::mbar_init(&t->q_full, 1);
    tc::mbar_init(&t->qsf_full, 2);
    tc::mbar_init(&t->drain, 1);
    t->abort = 0;
    tc::fence_mbar_init();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t taddr = t->taddr;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_tensormap(&keys);
      tc::prefetch_tensormap(&qmap);
      tc::mbar_arrive_expect_tx(&t->q_full, N * ROWB);
      tc::tma_load_2d(qbuf, &qmap, &t->q_full, 0, b * N);
      int issued = 0;
      for (int i = 0; i < ntile; ++i) {
        const int stage = i % C::STAGES, round = i / C::STAGES;
        if (!tc::mbar_wait(&t->empty[stage], (round & 1) ^ 1, abort)) break;
        tc::mbar_arrive_expect_tx(&t->full[stage], C::STAGE_BYTES);
        tc::tma_load_2d(stages + stage * C::STAGE_BYTES, &keys, &t->full[stage], 0,
                        static_cast<int>(bs * a.capacity + static_cast<int64_t>(t0 + i) * kTile));
        ++issued;
      }
      // every copy issued must land before the CTA's shared memory goes away
      for (int i = issued - C::STAGES > 0 ? issued - C::STAGES : 0; i < issued; ++i) {
        const int stage = i % C::STAGES, round = i / C::STAGES;
        tc::mbar_wait_drain(&t->full[stage], round & 1);
      }
      tc::mbar_wait_drain(&t->q_full, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ tcgen05.cp + MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_mxf4nvf4(kTile, N);
      const uint32_t q_addr = tc::smem_u32(qbuf);
      bool ok = tc::mbar_wait(&t->q_full, 0, abort) && tc::mbar_wait(&t->qsf_full, 0, abort);
      if (ok) {
        tc::tc_fence_after();
        for (int kk = 0; kk < C::KSTEPS; ++kk)
          tc::tmem_cp_32x128b_warpx4(taddr + sfb_col + kk * 4, tc::smem_desc_rows16(tc::smem_u32(qsf + kk * kSfBlock)));
      }
      for (int i = 0; ok && i < ntile; ++i) {
        const int stage = i % C::STAGES, round = i / C::STAGES;
        const int ab = i & 1, ra = i >> 1;
        if (!tc::mbar_wait(&t->full[stage], round & 1, abort)) break;
        if (!tc::mbar_wait(&t->sf_full[stage], round & 1, abort)) break;
        if (!tc::mbar_wait(&t->acc_empty[ab], (ra & 1) ^ 1, abort)) break;
        tc::tc_fence_after();
        const uint32_t a_addr = tc::smem_u32(stages + stage * C::STAGE_BYTES);
        const uint32_t sf_addr = tc::smem_u32(sfbuf + stage * C::SF_BYTES);
        const uint32_t sfa = taddr + sfa_col0 + ab * C::SF_COLS;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk)
          tc::tmem_cp_32x128b_warpx4(sfa + kk * 4, tc::smem_desc_rows16(sf_addr + kk * kSfBlock));
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
          const uint64_t adesc = tc::smem_desc(a_addr + kk * 32, 8 * ROWB, C::SWIZZLE);
          const uint64_t bdesc = tc::smem_desc(q_addr + kk * 32, 8 * ROWB, C::SWIZZLE);
          tc::mma_mxf4nvf4(taddr + acc_col0 + ab * N, adesc, bdesc, idesc, sfa + kk * 4, taddr + sfb_col + kk * 4,
                           kk > 0 ? 1u : 0u);
        }
        tc::tc_commit(&t->empty[stage]);
        tc::tc_commit(&t->acc_full[ab]);
      }
      // every tcgen05 operation issued must finish before tensor memory is released
      tc::tc_commit(&t->drain);
      tc::mbar_wait_drain(&t->drain, 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ scale-block builders (64 threads)
    const int tid = threadIdx.x - 64;
    // query scales: rows >= N (padding heads) are zero
    for (int r = tid; r < kTile; r += 64) {
      const uint8_t* src = a.q_scales + (static_cast<int64_t>(b) * N + r) * nblk;
      for (int kk = 0; kk < C::KSTEPS; ++kk) {
        const uint32_t w = r < N ? *reinterpret_cast<const uint32_t*>(src + kk * 4) : 0u;
        reinterpret_cast<uint32_t*>(qsf + kk * kSfBlock)[(r & 31) * 4 + (r >> 5)] = w;
      }
    }
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&t->qsf_full);
    // key scales: the global loads run kPf tiles ahead of the shared-memory
    // writes, so no tile waits for a memory round trip
    constexpr int kPf = 4;
    uint32_t pf[kPf][2][C::KSTEPS];
    auto load_scales = [&](int i, uint32_t (&w)[2][C::KSTEPS]) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int64_t s = static_cast<int64_t>(t0 + i) * kTile + tid + rr * 64;
        const uint32_t* src =
            reinterpret_cast<const uint32_t*>(a.idx_scales + (bs * a.capacity + s) * nblk);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) w[rr][kk] = (i < ntile && s < n_c) ? __ldg(src + kk) : 0u;
      }
    };
#pragma unroll
    for (int u = 0; u < kPf; ++u) load_scales(u, pf[u]);
    bool ok = true;
    for (int i0 = 0; ok && i0 < ntile; i0 += kPf) {
#pragma unroll
      for (int u = 0; u < kPf; ++u) {
        const int i = i0 + u;
        if (ok && i < ntile) {
          const int stage = i % C::STAGES, round = i / C::STAGES;
          ok = tc::mbar_wait(&t->empty[stage], (round & 1) ^ 1, abort);
          if (ok) {
            uint32_t* dst = reinterpret_cast<uint32_t*>(sfbuf + stage * C::SF_BYTES);
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int r = tid + rr * 64;
#pragma unroll
              for (int kk = 0; kk < C::KSTEPS; ++kk) dst[kk * (kSfBlock / 4) + (r & 31) * 4 + (r >> 5)] = pf[u][rr][kk];
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&t->sf_full[stage]);
            load_scales(i + kPf, pf[u]);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 4-11)
    // Two sets of four warps (one per 32-lane quarter of tensor memory): set s
    // takes the tiles of parity s, whose accumulator is buffer s.
    const int set = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;                  // tensor-memory lane == tile row
    const int et = threadIdx.x - 128;                     // 0 .. 255
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    for (int i = et; i < kBins; i += kEpiThreads) t->hist[i] = 0;
    epilogue_sync();
    float* out = a.scores + static_cast<int64_t>(b) * a.capacity;
    for (int i = set; i < ntile; i += 2) {
      const int ab = set, ra = i >> 1;
      if (!tc::mbar_wait(&t->acc_full[ab], ra & 1, abort)) break;
      tc::tc_fence_after();
      // sum_h w_h max(0, s_h), four partial sums
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = 0; c < N; c += 32) {
        uint32_t v[32];
        tc::tmem_ld32(taddr + lane_base + acc_col0 + ab * N + c, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 32; h += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(wsm + c + h);
          acc[0] = fmaf(w4.x, fmaxf(__uint_as_float(v[h]), 0.f), acc[0]);
          acc[1] = fmaf(w4.y, fmaxf(__uint_as_float(v[h + 1]), 0.f), acc[1]);
          acc[2] = fmaf(w4.z, fmaxf(__uint_as_float(v[h + 2]), 0.f), acc[2]);
          acc[3] = fmaf(w4.w, fmaxf(__uint_as_float(v[h + 3]), 0.f), acc[3]);
        }
      }
      const float score = (acc[0] + acc[1]) + (acc[2] + acc[3]);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&t->acc_empty[ab]);
      const int64_t s = static_cast<int64_t>(t0 + i) * kTile + row;
      if (s < n_c) out[s] = score;
      warp_hist_add(t->hist, score_key(score) >> 20, s < n_c);
    }
    epilogue_sync();
    uint32_t* gh = a.hist1 + static_cast<int64_t>(b) * kBins;
    for (int i = et; i < kBins; i += kEpiThreads)
      if (t->hist[i]) atomicAdd(&gh[i], t->hist[i]);
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(taddr, ncols);
  }
  if (threadIdx.x == 0 && t->abort) atomicOr(a.status, DSV4_STATUS_TIMEOUT);
}

// ------------------------------------------------------------------------------ host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_rows(CUtensorMap* map, const void* base, int rowbytes, int64_t rows, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rowbytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(rowbytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(rowbytes), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = rowbytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                : rowbytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int ROWB>
int launch_tc(const IndexTcArgs& a, const CUtensorMap& keys, const CUtensorMap& qmap, cudaStream_t st) {
  using C = TcCfg<ROWB>;
  size_t smem = 1024 + C::STAGES * (C::STAGE_BYTES + C::SF_BYTES) + ((a.N * ROWB + 1023) & ~1023) + C::SF_BYTES +
                sizeof(SmemTail) + 16 + a.N * 4;
  // keep at most two CTAs per SM so that their tensor-memory allocations always fit
  const size_t floor_bytes = a.tmem_cols > 256 ? 120 * 1024 : 80 * 1024;
  if (smem < floor_bytes) smem = floor_bytes;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(index_scores_tc_kernel<ROWB>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  });
  return launch_pdl(index_scores_tc_kernel<ROWB>, dim3(a.ctas_per_seq, a.B), dim3(kThreads), smem, st, keys, qmap, a);
}

}  // namespace

bool encode_u8_rows(CUtensorMap* map, const void* base, int64_t rows, int row_bytes, int box_bytes, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_index_scores_tc(const IndexTcArgs& a, const uint8_t* key_codes, const uint8_t* q_codes, cudaStream_t st) {
  const int rowb = a.Di / 2;
  CUtensorMap keys, qmap;
  if (!encode_rows(&keys, key_codes, rowb, static_cast<int64_t>(a.B / a.T) * a.capacity, kTile)) return DSV4_ERR_CUDA;
  if (!encode_rows(&qmap, q_codes, rowb, static_cast<int64_t>(a.B) * a.N, a.N)) return DSV4_ERR_CUDA;
  switch (rowb) {
    case 32: return launch_tc<32>(a, keys, qmap, st);
    case 64: return launch_tc<64>(a, keys, qmap, st);
    case 128: return launch_tc<128>(a, keys, qmap, st);
    default: return DSV4_ERR_UNSUPPORTED;
  }
}

}  // namespace dsv4
