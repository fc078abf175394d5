// CSA / HCA decode attention: one softmax over (selected or all) compressed
// entries together with the raw sliding-window tokens.
//
// vibecoco.ai, "DeepSeek V4 agent architecture", section
// "混合注意力：两种压缩，交替使用": CSA attends over the top-k compressed blocks
// plus a sliding-window branch of recent raw tokens; HCA attends densely over
// every compressed entry. pnsm.cn, "DeepSeek V4 架构深度解析…", section 2.1
// "CSA：压缩稀疏注意力": the window and the compressed KV feed one attention.
//
// Rows of sequence b are numbered: first the compressed entries (the top-k
// list for CSA, every entry for HCA), then the window tokens oldest first.
// attn_split_kernel gives each CTA a contiguous range of rows (a split) and
// all heads of a head group, runs an online softmax over it in fp32 and writes
// the normalised partial output with its log-sum-exp; attn_merge_kernel
// combines the splits: o = sum_s exp(lse_s - lse) o_s, lse = log sum_s exp(lse_s).
#include <mutex>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace dsv4 {

namespace {
constexpr int RT = 16;        // rows per tile
constexpr int NT = 256;       // threads per CTA
constexpr int HG = 64;        // max heads per CTA (head group)

// Value of element d of row r of sequence b (K or V side).
struct RowSrc {
  const uint8_t* nope;
  const float* scale;
  const uint16_t* rope;
  const uint16_t* win;
};
}  // namespace

// grid (splits, B, head groups), block 256.
// dynamic smem: q bf16 [HP][D], kT fp32 [D][RT], v fp32 [RT][Dv], s fp32 [HP][RT], row ids
template <int HP, int ACC>
__global__ void __launch_bounds__(NT) attn_split_kernel(AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smraw[];
  pdl_trigger();
  pdl_wait();
  constexpr int TPH = NT / HP;
  const int D = a.D, Dv = a.Dv;
  uint16_t* qs = reinterpret_cast<uint16_t*>(smraw);
  float* kT = reinterpret_cast<float*>(smraw + ((HP * D * 2 + 15) & ~15));
  float* vs = kT + D * RT;
  float* ss = vs + RT * Dv;
  int64_t* rowid = reinterpret_cast<int64_t*>(ss + HP * RT);   // >= 0: entry, < 0: -(window source row) - 1

  const int split = blockIdx.x, b = blockIdx.y;
  const int h0 = blockIdx.z * HG;
  const int tid = threadIdx.x;

  const int64_t n_tok = vseq_tokens(a.n_tokens, b, a.T);
  const int64_t bs = b / a.T;   // the sequence whose cache planes this (virtual) sequence reads
  const int64_t n_c = n_tok / a.ratio < a.capacity ? n_tok / a.ratio : a.capacity;
  const int64_t n_win = n_tok < a.window ? n_tok : a.window;
  const int64_t n_main = a.n_sel > 0 ? a.n_sel : (a.n_sel < 0 ? 0 : n_c);
  const int64_t R = n_main + n_win;
  const int64_t r0 = static_cast<int64_t>(split) * a.rows_per_split;
  int64_t r1 = r0 + a.rows_per_split;
  if (r1 > R) r1 = R;

  for (int i = tid; i < HP * D; i += NT) {
    const int h = h0 + i / D;
    qs[i] = h < a.H ? a.q[(static_cast<int64_t>(b) * a.H + h) * D + (i % D)] : 0;
  }

  const RowSrc K{a.k_nope, a.k_scale, a.k_rope, a.win_k};
  const RowSrc V = a.separate_v ? RowSrc{a.v_nope, a.v_scale, a.v_rope, a.win_v} : K;

  const int my_h = tid / TPH, my_u = tid % TPH;
  float m = -INFINITY, l = 0.f;
  float acc[ACC];
#pragma unroll
  for (int i = 0; i < ACC; ++i) acc[i] = 0.f;

  for (int64_t t0 = r0; t0 < r1; t0 += RT) {
    __syncthreads();
    if (tid < RT) {
      const int64_t r = t0 + tid;
      int64_t id = INT64_MIN;   // masked row
      if (r < r1) {
        if (r < n_main) {
          int64_t e = a.n_sel > 0 ? a.topk[static_cast<int64_t>(b) * a.n_sel + r] : r;
          if (e < -1 || e >= n_c) {
            atomicOr(a.status, DSV4_STATUS_BAD_INDEX);
            e = -1;
          }
          if (e >= 0) id = e;
        } else {
          const int64_t pos = n_tok - n_win + (r - n_main);
          id = a.span == 0 ? -(bs * a.window + pos % a.window) - 1
                           : -(bs * a.span + pos - (a.n_tokens[bs] - a.span)) - 1;
        }
      }
      rowid[tid] = id;
    }
    __syncthreads();
    // dequantise the tile: kT[d][r], vs[r][d]
    for (int i = tid; i < RT * D; i += NT) {
      const int r = i / D, d = i % D;
      const int64_t id = rowid[r];
      float kval = 0.f, vval = 0.f;
      if (id >= 0) {
        const int64_t e = bs * a.capacity + id;
        if (d < a.d_nope) {
          kval = e4m3_to_f32(K.nope[e * a.d_nope + d]) * K.scale[e];
          vval = a.separate_v ? e4m3_to_f32(V.nope[e * a.d_nope + d]) * V.scale[e] : kval;
        } else {
          kval = bf16_to_f32(K.rope[e * a.d_rope + (d - a.d_nope)]);
          vval = a.separate_v ? bf16_to_f32(V.rope[e * a.d_rope + (d - a.d_nope)]) : kval;
        }
      } else if (id != INT64_MIN) {
        const int64_t slot = -id - 1;
        kval = bf16_to_f32(K.win[slot * D + d]);
        vval = a.separate_v ? bf16_to_f32(V.win[slot * D + d]) : kval;
      }
      kT[d * RT + r] = kval;
      if (d < Dv) vs[r * Dv + d] = vval;
    }
    __syncthreads();
    // scores: thread -> row (tid % RT), heads tid / RT + 16 j
    {
      const int r = tid % RT;
      const bool valid = rowid[r] != INT64_MIN;
      for (int h = tid / RT; h < HP; h += NT / RT) {
        const uint16_t* qr = qs + h * D;
        float dot = 0.f;
        for (int d = 0; d < D; ++d) dot = fmaf(bf16_to_f32(qr[d]), kT[d * RT + r], dot);
        ss[h * RT + r] = valid ? dot * a.sm_scale : -INFINITY;
      }
    }
    __syncthreads();
    // online softmax + PV for (my_h, my dims)
    {
      const float* sr = ss + my_h * RT;
      float mx = m;
#pragma unroll
      for (int r = 0; r < RT; ++r) mx = fmaxf(mx, sr[r]);
      if (mx != -INFINITY) {
        const float alpha = expf(m - mx);   // m = -inf -> 0
        float p[RT];
        float psum = 0.f;
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          p[r] = expf(sr[r] - mx);
          psum += p[r];
        }
        l = l * alpha + psum;
        m = mx;
#pragma unroll
        for (int i = 0; i < ACC; ++i) {
          const int d = my_u + TPH * i;
          float v = acc[i] * alpha;
          if (d < Dv) {
#pragma unroll
            for (int r = 0; r < RT; ++r) v = fmaf(p[r], vs[r * Dv + d], v);
          }
          acc[i] = v;
        }
      }
    }
  }
  const int h = h0 + my_h;
  if (h < a.H && my_h < HP) {
    const int64_t base = (static_cast<int64_t>(b) * a.H + h) * a.splits + split;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int i = 0; i < ACC; ++i) {
      const int d = my_u + TPH * i;
      if (d < Dv) a.part_o[base * Dv + d] = acc[i] * inv;
    }
    if (my_u == 0) a.part_lse[base] = l > 0.f ? m + logf(l) : -INFINITY;
  }
}

// grid (B * H, ceil(Dv / 128)), block 128: one (sequence, head) and 128 dims
// per CTA. Warp g sums splits g, g + 4, ... for 4 dims per lane, with several
// splits' loads in flight; the four warps' sums are then added.
__global__ void __launch_bounds__(128) attn_merge_kernel(AttnArgs a) {
  pdl_trigger();
  pdl_wait();
  const int64_t bh = blockIdx.x;
  const float* lse = a.part_lse + bh * a.splits;
  const int sg = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float mx = -INFINITY;
  for (int s = lane; s < a.splits; s += 32) mx = fmaxf(mx, lse[s]);
  mx = warp_max(mx);
  float tot = 0.f;
  if (mx != -INFINITY)
    for (int s = lane; s < a.splits; s += 32) tot += expf(lse[s] - mx);
  tot = warp_sum(tot);
  const int d0 = blockIdx.y * 128 + lane * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tot > 0.f && d0 < a.Dv) {
    const float* po = a.part_o + bh * a.splits * a.Dv + d0;
#pragma unroll 4
    for (int s = sg; s < a.splits; s += 4) {
      const float w = expf(lse[s] - mx);
      const float4 v = *reinterpret_cast<const float4*>(po + static_cast<int64_t>(s) * a.Dv);
      if (w > 0.f) {   // a split without rows may leave its partial unwritten
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
  }
  __shared__ float4 red[4][32];
  red[sg][lane] = acc;
  __syncthreads();
  if (sg == 0 && d0 < a.Dv) {
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    const float4 r1 = red[1][lane], r2 = red[2][lane], r3 = red[3][lane];
    *reinterpret_cast<float4*>(a.out + bh * a.Dv + d0) =
        make_float4(((acc.x + r1.x) + (r2.x + r3.x)) * inv, ((acc.y + r1.y) + (r2.y + r3.y)) * inv,
                    ((acc.z + r1.z) + (r2.z + r3.z)) * inv, ((acc.w + r1.w) + (r2.w + r3.w)) * inv);
  }
  if (threadIdx.x == 0 && blockIdx.y == 0 && a.lse) a.lse[bh] = tot > 0.f ? mx + logf(tot) : -INFINITY;
}

// Merge of the tensor-core kernel's splits: partials are f16 [B][splits][head
// groups][D][64 heads] (each normalised to a convex combination of its rows;
// in each 128-byte row of a dim d the 16-byte granule of heads 8q .. 8q + 7
// sits at granule q ^ (d & 7)), with two fp32 log sums [B][H][splits] each:
// lse_s, of the split's softmax weights, and lse'_s, of the scale of its
// partial, so that out = sum_s exp(lse'_s) o_s / sum_s exp(lse_s).
// grid (B * head groups, D / KD), block 256: KD dims x 64 heads per CTA;
// thread t takes split group t / (8 KD) (splits s = group mod KSG), dim
// t / 8 % KD and heads 8 (t % 8) .. + 7. Per pass of up to KS splits every
// thread issues its partial loads and its share of the log-sum-exps at once
// (one round trip); the split weights exp(lse - max) are computed once per
// CTA, each thread accumulates its splits and the split groups are summed in
// shared memory. With more than KS splits the passes rescale the running result.
// KS splits per pass in KSG groups of threads; each CTA merges KD dims of one
// sequence and head group (KSG * KD * 8 = 256 threads: split group, dim, 8 heads).
// Many splits: (64, 4, 8); a few (at most 8, the batched CSA plan): (8, 1, 32),
// so that the CTAs are fewer, lighter and all resident at once.
template <int KS, int KSG, int KD>
__global__ void __launch_bounds__(256, KS <= 8 ? 4 : 2) attn_merge_tc_kernel(AttnArgs a) {
  constexpr int kT = 256;
  constexpr int kS = KS;   // splits per pass
  constexpr int kSg = KSG; // split groups
  constexpr int kU = kS / kSg;
  constexpr int kL = 64 * kS / kT;   // log-sum-exps each thread stages per pass
  static_assert(KSG * KD * 8 == kT, "one thread per (split group, dim, 8 heads)");
  pdl_trigger();
  pdl_wait();
  const int hgs = (a.H + 63) / 64;
  const int b = blockIdx.x / hgs, hg = blockIdx.x % hgs;
  const int h0 = hg * 64;
  const int hcount = a.H - h0 < 64 ? a.H - h0 : 64;
  __shared__ float s_lse[64][kS + 1];                   // [head][split]
  __shared__ __align__(16) float s_w[kS][64 + 4];       // [split][head]: partial weights relative to the running max
  __shared__ float s_m[64], s_l[64], s_r[64];           // running max and sum per head, rescale of this pass
  __shared__ float s_acc[kSg][64][KD + 1];
  const int t = threadIdx.x;
  const int sg = t / (8 * KD), dl = (t >> 3) % KD, hq = (t & 7) * 8;
  const int d = blockIdx.y * KD + dl;
  const float* lse0 = a.part_lse + (static_cast<int64_t>(b) * a.H + h0) * a.splits;
  const float* lsev0 = a.part_lsev + (static_cast<int64_t>(b) * a.H + h0) * a.splits;
  // granule hq / 8 of dim d sits at granule (hq / 8) ^ (d & 7) of the row
  const int dd0 = d < a.D ? d : 0;
  const uint16_t* part = reinterpret_cast<const uint16_t*>(a.part_o) +
                         ((static_cast<int64_t>(b) * a.splits * hgs + hg) * a.D + dd0) * 64 + (((hq >> 3) ^ (dd0 & 7)) << 3);
  const int64_t sstride = static_cast<int64_t>(hgs) * a.D * 64;   // between splits
  if (t < 64) {
    s_m[t] = -INFINITY;
    s_l[t] = 0.f;
  }
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int s0 = 0; s0 < a.splits; s0 += kS) {
    const int ns = a.splits - s0 < kS ? a.splits - s0 : kS;
    uint4 v[kU];
    float lv[kL], lvv[kL];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int s = sg + kSg * u;
      v[u] = s < ns ? __ldcg(reinterpret_cast<const uint4*>(part + (s0 + s) * sstride)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kL; ++u) {
      const int i = t + u * kT, h = i / kS, s = i % kS;
      const bool in = h < hcount && s < ns;
      lv[u] = in ? __ldcg(lse0 + static_cast<int64_t>(h) * a.splits + s0 + s) : -INFINITY;
      lvv[u] = in ? __ldcg(lsev0 + static_cast<int64_t>(h) * a.splits + s0 + s) : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < kL; ++u) {
      const int i = t + u * kT;
      s_lse[i / kS][i % kS] = lv[u];
      s_w[i % kS][i / kS] = lvv[u];     // lse', turned into the output weight below
    }
    __syncthreads();
    {
      // head t / 4: this pass's max and sum of exp (four threads, every fourth split)
      const int h = t >> 2, part4 = t & 3;
      float mx = -INFINITY;
      for (int s = part4; s < ns; s += 4) mx = fmaxf(mx, s_lse[h][s]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mo = s_m[h], mn = fmaxf(mo, mx);
      float sum = 0.f;
      for (int s = part4; s < ns; s += 4) {
        // weights relative to the running max: of the normaliser (w) and of the
        // split's partial (u); a split without rows gets 0
        const float x = s_lse[h][s];
        const float w = x == -INFINITY ? 0.f : __expf(x - mn);
        const float u = x == -INFINITY ? 0.f : __expf(s_w[s][h] - mn);
        s_w[s][h] = u;
        sum += w;
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      if (part4 == 0) {
        const float r = mo == -INFINITY ? 0.f : __expf(mo - mn);
        s_r[h] = r;
        s_l[h] = s_l[h] * r + sum;
        s_m[h] = mn;
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] *= s_r[hq + i];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int s = sg + kSg * u;
      if (s < ns) {
        const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        const float4 wa = *reinterpret_cast<const float4*>(&s_w[s][hq]);
        const float4 wb = *reinterpret_cast<const float4*>(&s_w[s][hq + 4]);
        const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint16_t bits = static_cast<uint16_t>((i & 1) ? w4[i >> 1] >> 16 : w4[i >> 1] & 0xFFFFu);
          // a split without rows may have left its partial unwritten
          acc[i] = w[i] > 0.f ? fmaf(w[i], __half2float(__ushort_as_half(bits)), acc[i]) : acc[i];
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) s_acc[sg][hq + i][dl] = acc[i];
  __syncthreads();
  for (int o = t; o < 64 * KD; o += kT) {
    const int r = o / KD, dd = o % KD;   // head r, dim dd of the CTA's KD
    if (r < hcount) {
      float sum;
      if (KSG == 4) sum = (s_acc[0][r][dd] + s_acc[1][r][dd]) + (s_acc[2][r][dd] + s_acc[3][r][dd]);
      else sum = s_acc[0][r][dd];
      const float L = s_l[r];
      const int dg = blockIdx.y * KD + dd;
      if (dg < a.D) a.out[(static_cast<int64_t>(b) * a.H + h0 + r) * a.Dv + dg] = L > 0.f ? sum / L : 0.f;
      if (blockIdx.y == 0 && dd == 0 && a.lse)
        a.lse[static_cast<int64_t>(b) * a.H + h0 + r] = L > 0.f ? s_m[r] + logf(L) : -INFINITY;
    }
  }
}

namespace {
template <int HP, int ACC>
int launch_split(const AttnArgs& a, dim3 grid, size_t smem, cudaStream_t st) {
  static std::once_flag flag;
  std::call_once(flag, [] {
    cudaFuncSetAttribute(attn_split_kernel<HP, ACC>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  });
  return launch_pdl(attn_split_kernel<HP, ACC>, grid, dim3(NT), smem, st, a);
}
}  // namespace

int launch_attention(const AttnArgs& a, int head_groups, cudaStream_t st) {
  const int hp = a.H >= 64 ? 64 : (a.H > 16 ? 32 : 16);
  const int tph = NT / hp;
  const int need = (a.Dv + tph - 1) / tph;
  const size_t smem = ((static_cast<size_t>(hp) * a.D * 2 + 15) & ~static_cast<size_t>(15)) +
                      (static_cast<size_t>(a.D) * RT + RT * a.Dv + hp * RT) * sizeof(float) + RT * sizeof(int64_t);
  const dim3 grid(a.splits, a.B, head_groups);
  int e;
  if (hp == 16)
    e = need <= 8 ? launch_split<16, 8>(a, grid, smem, st)
        : need <= 16 ? launch_split<16, 16>(a, grid, smem, st) : launch_split<16, 36>(a, grid, smem, st);
  else if (hp == 32)
    e = need <= 16 ? launch_split<32, 16>(a, grid, smem, st)
        : need <= 32 ? launch_split<32, 32>(a, grid, smem, st) : launch_split<32, 72>(a, grid, smem, st);
  else
    e = need <= 32 ? launch_split<64, 32>(a, grid, smem, st)
        : need <= 64 ? launch_split<64, 64>(a, grid, smem, st) : launch_split<64, 144>(a, grid, smem, st);
  if (e) return e;
  return launch_attention_merge(a, st);
}

int launch_attention_merge_tc(const AttnArgs& a, int head_groups, cudaStream_t st) {
  if (a.splits <= 8)
    return launch_pdl(attn_merge_tc_kernel<8, 1, 32>, dim3(a.B * head_groups, (a.D + 31) / 32), dim3(256), 0, st, a);
  return launch_pdl(attn_merge_tc_kernel<64, 4, 8>, dim3(a.B * head_groups, (a.D + 7) / 8), dim3(256), 0, st, a);
}

int launch_attention_merge(const AttnArgs& a, cudaStream_t st) {
  return launch_pdl(attn_merge_kernel, dim3(a.B * a.H, (a.Dv + 127) / 128), dim3(128), 0, st, a);
}

}  // namespace dsv4
