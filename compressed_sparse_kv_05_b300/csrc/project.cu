// Projection of the compressor's input streams from hidden states, with RoPE,
// on the 5th-generation tensor cores (tcgen05 kind::f16, bf16 operands, fp32
// accumulators in tensor memory).
//
// vibecoco.ai, "DeepSeek V4 agent architecture", section
// "混合注意力：两种压缩，交替使用": the pooling is learned, so the token keys x,
// their gate logits z, the indexer keys u and their gate logits zu are linear
// projections of the token's hidden state. devpress.csdn.net,
// "DeepSeek-V4：百万Token上下文，这次智能体真的能用了", section
// "二、DeepSeek-V4的核心架构创新", part "位置编码的长度泛化优化": positions enter
// through RoPE. Reading: the standard rotation, pair (2i, 2i + 1) of the
// rotated dims turning by pos * base^(-2i/d), on the trailing d_rope dims of x
// and the trailing min(d_rope, Di) dims of u, at the token's absolute position.
//
// C[M][N] = H[M][K] . W[N][K]^T with M = B * T token rows, K the hidden size
// and N = 2 D + 2 Di output columns (W's rows: x, z, u, zu). Tiles of 128 rows
// x bn columns (bn of 128 .. 256 chosen per call so that the tiles fill the
// SMs' waves); K in steps of 64 (128-byte rows, 128-byte swizzle) through a
// 4-stage TMA ring; one thread issues 4 MMAs (M = 128, N = bn, K = 16) per
// step into one of two accumulators (256 tensor-memory columns each), so the
// epilogue of one tile overlaps the MMAs of the next. Persistent CTAs take
// tiles column-block first, so the CTAs working at one time share their
// hidden-state rows in L2 (the weights stay L2-resident).
//
// Epilogue (warps 2-5, warp w reading tensor-memory lanes 32 (w % 4) ...):
// per 32-column chunk, the fp32 accumulators of one row; rotated columns turn
// by the row's angle, computed without losing the position's bits: with t_i =
// theta_i / pi held as a float pair (hi + lo), pos * t_i = p + e exactly (p =
// fl(pos * hi), e from an fma) plus pos * lo; p is reduced modulo 2 exactly,
// and sincospi gives the sine and cosine of pi times the remainder. Each
// value is rounded once to bf16 and stored to its stream.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace dsv4 {

namespace {

constexpr int kPM = 128;                       // rows per tile (MMA M)
constexpr int kPN = 256;                       // columns per tile (MMA N)
constexpr int kPK = 64;                        // hidden dims per stage (128 bytes of bf16)
constexpr int kPStages = 4;
constexpr int kPThreads = 192;                 // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kPABytes = kPM * kPK * 2;        // 16 KB
constexpr int kPBBytes = kPN * kPK * 2;        // 32 KB
constexpr int kPStageBytes = kPABytes + kPBBytes;
constexpr uint32_t kPCols = 2 * kPN;           // two accumulators

struct ProjTail {
  uint64_t full[kPStages], empty[kPStages], acc_full[2], acc_empty[2], drain;
  uint32_t taddr;
  int abort;
};

// bf16 with both operands K-major, fp32 accumulator (the f16 descriptor with
// the A and B formats set to bf16)
DSV4_DEV uint32_t idesc_bf16(uint32_t N) { return tc::idesc_f16_f32(kPM, N, 0, 0) | (1u << 7) | (1u << 10); }

// the row's position (n_tokens of its sequence before this call, plus its token index)
DSV4_DEV float row_position(const ProjArgs& a, int row) {
  const int b = row / a.T, t = row % a.T;
  return static_cast<float>(a.n_tokens[b] + t);
}

// Rotate 16 pairs of v (32 consecutive columns, pair j = (v[2j], v[2j + 1]))
// whose first pair is pair i0 of the table (hi, lo).
DSV4_DEV void rope32(float* v, float pos, const float* hi, const float* lo, int i0) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float th = hi[i0 + j], tl = lo[i0 + j];
    const float p = pos * th;
    const float e = fmaf(pos, th, -p);                 // pos * th = p + e exactly
    const float r = (p - 2.f * rintf(0.5f * p)) + fmaf(pos, tl, e);
    float s, c;
    sincospif(r, &s, &c);
    const float x0 = v[2 * j], x1 = v[2 * j + 1];
    v[2 * j] = x0 * c - x1 * s;
    v[2 * j + 1] = x0 * s + x1 * c;
  }
}

}  // namespace

__global__ void __launch_bounds__(kPThreads, 1)
    project_kernel(const __grid_constant__ CUtensorMap hmap, const __grid_constant__ CUtensorMap wmap,
                   const __grid_constant__ ProjArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* stages =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  ProjTail* t = reinterpret_cast<ProjTail*>(stages + kPStages * kPStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &t->abort;
  pdl_trigger();
  if (threadIdx.x == 0) {
    tc::prefetch_tensormap(&hmap);
    tc::prefetch_tensormap(&wmap);
  }
  if (warp == 1) tc::tmem_alloc(&t->taddr, kPCols);
  if (threadIdx.x == 32) {
    for (int s = 0; s < kPStages; ++s) {
      tc::mbar_init(&t->full[s], 1);
      tc::mbar_init(&t->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&t->acc_full[b], 1);
      tc::mbar_init(&t->acc_empty[b], 4);
    }
    tc::mbar_init(&t->drain, 1);
    t->abort = 0;
    tc::fence_mbar_init();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t taddr = t->taddr;
  const int ksteps = a.K / kPK;
  // the hidden states may be written by the kernel before this one (the
  // weights too, in principle): every load after the wait
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0;   // stage uses so far
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < a.tiles; tile += gridDim.x) {
        const int mt = tile / a.tiles_n, nt = tile % a.tiles_n;
        for (int ks = 0; ks < ksteps; ++ks, ++g) {
          const int s = g % kPStages, round = g / kPStages;
          if (!(ok = tc::mbar_wait(&t->empty[s], (round & 1) ^ 1, abort))) break;
          unsigned char* st = stages + s * kPStageBytes;
          tc::mbar_arrive_expect_tx(&t->full[s], kPABytes + a.bn * kPK * 2);
          tc::tma_load_2d(st, &hmap, &t->full[s], ks * kPK, mt * kPM);
          tc::tma_load_2d(st + kPABytes, &wmap, &t->full[s], ks * kPK, nt * a.bn);
        }
      }
      // every copy issued must land before the CTA's shared memory goes away
      for (int i = g - kPStages > 0 ? g - kPStages : 0; i < g; ++i)
        tc::mbar_wait_drain(&t->full[i % kPStages], (i / kPStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int g = 0, j = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16(static_cast<uint32_t>(a.bn));
      for (int tile = blockIdx.x; ok && tile < a.tiles; tile += gridDim.x, ++j) {
        const int buf = j & 1, use = j >> 1;
        if (!(ok = tc::mbar_wait(&t->acc_empty[buf], (use & 1) ^ 1, abort))) break;
        tc::tc_fence_after();
        const uint32_t acc = taddr + buf * kPN;
        for (int ks = 0; ks < ksteps; ++ks, ++g) {
          const int s = g % kPStages, round = g / kPStages;
          if (!(ok = tc::mbar_wait(&t->full[s], round & 1, abort))) break;
          tc::tc_fence_after();
          const uint32_t a_sa = tc::smem_u32(stages + s * kPStageBytes);
          const uint32_t b_sa = a_sa + kPABytes;
#pragma unroll
          for (int kk = 0; kk < kPK / 16; ++kk) {
            const uint64_t ad = tc::smem_desc(a_sa + kk * 32, 1024, tc::kSwizzle128B);
            const uint64_t bd = tc::smem_desc(b_sa + kk * 32, 1024, tc::kSwizzle128B);
            tc::mma_f16(acc, ad, bd, idesc, (ks | kk) ? 1u : 0u);
          }
          tc::tc_commit(&t->empty[s]);
        }
        if (!ok) break;
        tc::tc_commit(&t->acc_full[buf]);
      }
      // every MMA issued must finish before tensor memory is released
      tc::tc_commit(&t->drain);
      tc::mbar_wait_drain(&t->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5)
    const int q = warp & 3;                                  // tensor-memory lane quarter
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int D = a.d_nope + a.d_rope;
    int j = 0;
    for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x, ++j) {
      const int buf = j & 1, use = j >> 1;
      if (!tc::mbar_wait(&t->acc_full[buf], use & 1, abort)) break;
      tc::tc_fence_after();
      const int mt = tile / a.tiles_n, nt = tile % a.tiles_n;
      const int row = mt * kPM + q * 32 + lane;
      const bool live = row < a.M;
      const float pos = live ? row_position(a, live ? row : 0) : 0.f;
      for (int c = 0; c < a.bn / 32; ++c) {
        uint32_t raw[32];
        tc::tmem_ld32(taddr + lane_off + buf * kPN + c * 32, raw);
        tc::tmem_wait_ld();
        const int n0 = nt * a.bn + c * 32;                   // first output column of the chunk
        if (!live || n0 >= a.N) continue;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]);
        uint16_t* dst;
        if (n0 < D) {                                        // x: rotated from d_nope on
          if (n0 >= a.d_nope) rope32(v, pos, a.rx_hi, a.rx_lo, (n0 - a.d_nope) / 2);
          dst = a.x + static_cast<int64_t>(row) * D + n0;
        } else if (n0 < 2 * D) {
          dst = a.z + static_cast<int64_t>(row) * D + (n0 - D);
        } else if (n0 < 2 * D + a.Di) {                      // u: rotated over its last ur dims
          const int cu = n0 - 2 * D;
          if (cu >= a.Di - a.ur) rope32(v, pos, a.ru_hi, a.ru_lo, (cu - (a.Di - a.ur)) / 2);
          dst = a.u + static_cast<int64_t>(row) * a.Di + cu;
        } else {
          dst = a.zu + static_cast<int64_t>(row) * a.Di + (n0 - 2 * D - a.Di);
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = static_cast<uint32_t>(f32_to_bf16(v[2 * i])) | (static_cast<uint32_t>(f32_to_bf16(v[2 * i + 1])) << 16);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&t->acc_empty[buf]);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(taddr, kPCols);
  }
  if (threadIdx.x == 0 && t->abort) atomicOr(a.status, DSV4_STATUS_TIMEOUT);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 map_encoder() {
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

// rows x K bf16 matrix (row stride K), boxes of box_rows rows x 64 columns, 128-byte swizzle
bool encode_bf16_rows(CUtensorMap* map, const void* base, int64_t rows, int K, int box_rows) {
  auto enc = map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kPK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// theta_i / pi = base^(-2i/d) / pi for i < d/2 as float pairs (hi, lo)
void rope_table(double base, int d, float* hi, float* lo) {
  for (int i = 0; i < d / 2; ++i) {
    const double v = std::pow(base, -2.0 * i / d) / 3.141592653589793238462643383279502884;
    hi[i] = static_cast<float>(v);
    lo[i] = static_cast<float>(v - static_cast<double>(hi[i]));
  }
}

}  // namespace

size_t project_smem_bytes() { return 1024 + static_cast<size_t>(kPStages) * kPStageBytes + sizeof(ProjTail); }

int launch_project(ProjArgs a, const void* hidden, const void* weight, double rope_base, int sms, cudaStream_t st) {
  // Tile width: the one of 256, 224, 192, 160, 128 columns with the least
  // time over all waves of tiles (tiles of one wave run side by side), so that
  // the last wave is not left nearly empty. A tile takes time in proportion to
  // bn + 218: its own columns plus a fixed part (the 128 hidden rows it loads,
  // the MMA issue, the epilogue) measured worth about 218 columns.
  const int tiles_m = (a.M + kPM - 1) / kPM;
  int best = kPN;
  int64_t best_cost = -1;
  for (int bn = kPN; bn >= 128; bn -= 32) {
    const int64_t tiles = static_cast<int64_t>(tiles_m) * ((a.N + bn - 1) / bn);
    const int64_t cost = ((tiles + sms - 1) / sms) * (bn + 218);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  a.bn = best;
  CUtensorMap hmap, wmap;
  if (!encode_bf16_rows(&hmap, hidden, a.M, a.K, kPM) || !encode_bf16_rows(&wmap, weight, a.N, a.K, a.bn))
    return DSV4_ERR_CUDA;
  rope_table(rope_base, a.d_rope, a.rx_hi, a.rx_lo);
  rope_table(rope_base, a.ur, a.ru_hi, a.ru_lo);
  a.tiles_n = (a.N + a.bn - 1) / a.bn;
  a.tiles = tiles_m * a.tiles_n;
  const int grid = a.tiles < sms ? a.tiles : sms;
  const size_t smem = project_smem_bytes();
  static std::once_flag once;
  std::call_once(once, [smem] {
    cudaFuncSetAttribute(project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  });
  return launch_pdl(project_kernel, dim3(grid), dim3(kPThreads), smem, st, hmap, wmap, a);
}

}  // namespace dsv4
