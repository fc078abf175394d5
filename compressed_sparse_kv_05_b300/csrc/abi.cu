// extern "C" entry points of libdsv4 (declared in include/dsv4.h): argument
// validation on the host, workspace carving, kernel launches on the caller's
// stream. No entry point allocates or frees device memory.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/dsv4.h"
#include "kernels.h"
#include "launch.cuh"

namespace dsv4 {
namespace {

constexpr int kTcTile = 128;            // rows per tile of the tensor-core attention, at most
constexpr int kTcMinTile = 32;          // and at least
constexpr int kTcMaxTiles = 8;          // tiles per CTA of the tensor-core attention, at most
constexpr int kRowTile = 16;
constexpr int kHeadGroup = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Streaming multiprocessors of the current device, queried once per device
// (148 on a B300; also the answer when no device can be queried, so that the
// host-side plans stay defined without a GPU). Grids are sized from it.
int sm_count() {
  constexpr int kMaxDevices = 64;
  constexpr int kDefault = 148;
  static std::mutex mu;
  static int count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return kDefault;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = kDefault;
    }
    count[dev] = n;
  }
  return count[dev];
}

int check_desc(const dsv4_layer_desc* d) {
  if (!d) return DSV4_ERR_INVALID_ARG;
  if (d->batch < 1 || d->capacity < 1 || d->d_nope < 0 || d->d_rope < 0 || d->ratio < 1 || d->window < 0 ||
      d->idx_dim < 0)
    return DSV4_ERR_INVALID_ARG;
  if (d->d_nope < 16 || d->d_nope > 512 || d->d_nope % 16) return DSV4_ERR_UNSUPPORTED;
  if (d->d_rope > 128 || d->d_rope % 8) return DSV4_ERR_UNSUPPORTED;
  if (d->d_nope + d->d_rope > 576) return DSV4_ERR_UNSUPPORTED;
  if (d->ratio > 256 || d->window > 4096) return DSV4_ERR_UNSUPPORTED;
  if (d->idx_dim && d->idx_dim != 64 && d->idx_dim != 128 && d->idx_dim != 256) return DSV4_ERR_UNSUPPORTED;
  return DSV4_OK;
}

#define DSV4_REQ(p)                                      \
  do {                                                   \
    if (!(p)) return DSV4_ERR_INVALID_ARG;               \
    if (!aligned16(p)) return DSV4_ERR_MISALIGNED;       \
  } while (0)

int check_kv_planes(const dsv4_kv_planes& p, const dsv4_layer_desc* d) {
  DSV4_REQ(p.nope);
  DSV4_REQ(p.scale);
  if (d->d_rope) DSV4_REQ(p.rope);
  return DSV4_OK;
}

int check_cache_read(const dsv4_layer_desc* d, const dsv4_cache* c) {
  if (!c) return DSV4_ERR_INVALID_ARG;
  int e = check_kv_planes(c->k, d);
  if (e) return e;
  if (d->separate_v && (e = check_kv_planes(c->v, d))) return e;
  if (d->window) {
    DSV4_REQ(c->win_k);
    if (d->separate_v) DSV4_REQ(c->win_v);
  }
  DSV4_REQ(c->n_tokens);
  DSV4_REQ(c->status);
  return DSV4_OK;
}

struct AttnPlan {
  int head_groups, splits, rows_per_split, tile_rows, tiles_per_split;
  bool tc;
  size_t part_bytes;   // bytes of the split partials (the log-sum-exps follow)
  size_t ws_bytes;
};

// n_sel: top-k width (CSA), 0 for every entry (HCA), < 0 for none (window only).
// T: queries per sequence (the call attends for batch * T virtual sequences).
AttnPlan attn_plan(const dsv4_layer_desc* d, int H, int n_sel, int T = 1) {
  AttnPlan p{};
  const int sms = sm_count();
  const int64_t nb = static_cast<int64_t>(d->batch) * T;
  p.head_groups = (H + kHeadGroup - 1) / kHeadGroup;
  const int64_t n_main = n_sel > 0 ? n_sel : (n_sel < 0 ? 0 : d->capacity);
  const int64_t rmax = n_main + d->window;
  const size_t Dv = static_cast<size_t>(d->d_nope + d->d_rope);
  p.tc = attention_tc_supported(H, d->d_nope, d->d_rope, d->separate_v);
  if (p.tc) {
    // Tiles of R rows (compressed rows, then window tokens, never mixed): the
    // largest R in {128, 64, 32} whose halving would still fit one wave of
    // CTAs is halved, so short row sets spread over more SMs; then runs of
    // consecutive tiles are spread evenly over one wave (one CTA per SM).
    const int64_t units = nb * p.head_groups;
    auto tiles_for = [&](int64_t r) { return (n_main + r - 1) / r + (d->window + r - 1) / r; };
    int64_t tr = kTcTile;
    while (tr > kTcMinTile && units * tiles_for(tr / 2) <= sms) tr /= 2;
    const int64_t tiles = tiles_for(tr);
    int64_t per_cta = (tiles * units + sms - 1) / sms;
    if (per_cta > kTcMaxTiles) per_cta = kTcMaxTiles;   // a CTA keeps its rows' sources in shared memory
    if (per_cta < 1) per_cta = 1;
    p.tile_rows = static_cast<int>(tr);
    p.tiles_per_split = static_cast<int>(per_cta);
    p.rows_per_split = static_cast<int>(per_cta * tr);
    p.splits = static_cast<int>((tiles + per_cta - 1) / per_cta);
    if (p.splits < 1) p.splits = 1;
    // f16 partials [B][splits][head groups][D][64], then two fp32 log sums [B][H][splits] each
    p.part_bytes = (static_cast<size_t>(nb) * p.splits * p.head_groups * Dv * 64 * 2 + 255) & ~size_t(255);
    p.ws_bytes = p.part_bytes + 2 * static_cast<size_t>(nb) * H * p.splits * sizeof(float) + 256;
    return p;
  }
  const int64_t want = (2 * sms + nb * p.head_groups - 1) / (nb * p.head_groups);
  const int64_t max_splits = (rmax + kRowTile - 1) / kRowTile;
  int64_t s = want < max_splits ? want : max_splits;
  if (s < 1) s = 1;
  int64_t rps = (rmax + s - 1) / s;
  rps = (rps + kRowTile - 1) / kRowTile * kRowTile;
  s = (rmax + rps - 1) / rps;
  if (s < 1) s = 1;
  p.splits = static_cast<int>(s);
  p.rows_per_split = static_cast<int>(rps);
  p.part_bytes = (static_cast<size_t>(nb) * H * p.splits * Dv * sizeof(float) + 255) & ~size_t(255);
  p.ws_bytes = static_cast<size_t>(nb) * H * p.splits * (Dv + 1) * sizeof(float) + 256;
  return p;
}

int index_heads_padded(int Hi) { return Hi <= 64 ? 64 : 128; }

struct IndexWs {
  size_t q_codes, q_scales, scores, hist1, hist2, cnt, above, cand, total;
};

// T: queries per sequence (batch * T virtual sequences, each with its own
// query, scores and selection).
IndexWs index_ws(const dsv4_layer_desc* d, int Hi, int k, int T = 1) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t N = index_heads_padded(Hi);
  const size_t B = static_cast<size_t>(d->batch) * T, cap = d->capacity;
  IndexWs w{};
  w.q_codes = 0;
  w.q_scales = up(w.q_codes + B * N * (d->idx_dim / 2));
  w.scores = up(w.q_scales + B * N * (d->idx_dim / 16));
  w.hist1 = up(w.scores + B * cap * sizeof(float));
  w.hist2 = up(w.hist1 + B * 4096 * sizeof(uint32_t));
  w.cnt = up(w.hist2 + B * 4096 * sizeof(uint32_t));
  w.above = up(w.cnt + B * kCntWords * sizeof(uint32_t));
  w.cand = up(w.above + B * static_cast<size_t>(k) * sizeof(int32_t));
  w.total = up(w.cand + B * cap * sizeof(uint64_t));
  return w;
}

size_t index_ws_bytes(const dsv4_layer_desc* d, int Hi, int k, int T = 1) { return index_ws(d, Hi, k, T).total; }

template <typename F>
void set_smem_once(std::once_flag& flag, F func, int bytes) {
  std::call_once(flag, [&] { cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes); });
}

int launch_status() { return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA; }

// n_sel: the top-k width (CSA), 0 for every entry (HCA), -1 for no compressed
// entry at all (a window-only CSA call, k = 0). T queries per sequence; with
// span_k the window tokens come from that span of the last T + W - 1 raw
// tokens of each sequence instead of the cache's ring.
int decode_common(const dsv4_layer_desc* d, const dsv4_cache* c, int H, const uint16_t* q, float sm_scale,
                  const int32_t* topk, int n_sel, float* out, float* lse, void* ws, size_t ws_bytes, void* stream,
                  int T = 1, const uint16_t* span_k = nullptr, const uint16_t* span_v = nullptr) {
  int e = check_desc(d);
  if (e) return e;
  if ((e = check_cache_read(d, c))) return e;
  if (H < 1 || T < 1) return DSV4_ERR_INVALID_ARG;
  if (H > 128) return DSV4_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->batch) * T > 65535) return DSV4_ERR_UNSUPPORTED;   // the grid's y extent
  DSV4_REQ(q);
  DSV4_REQ(out);
  DSV4_REQ(ws);
  if (lse && !aligned16(lse)) return DSV4_ERR_MISALIGNED;
  if (!(sm_scale == sm_scale)) return DSV4_ERR_INVALID_ARG;
  const bool span = T > 1 || span_k;
  if (span && d->window) {
    DSV4_REQ(span_k);
    if (d->separate_v) DSV4_REQ(span_v);
  }
  const AttnPlan p = attn_plan(d, H, n_sel, T);
  if (ws_bytes < p.ws_bytes) return DSV4_ERR_WORKSPACE;
  AttnArgs a{};
  a.B = d->batch * T; a.T = T; a.span = span ? T + d->window - 1 : 0;
  a.H = H; a.D = d->d_nope + d->d_rope; a.Dv = a.D; a.d_nope = d->d_nope; a.d_rope = d->d_rope;
  a.ratio = d->ratio; a.window = d->window; a.capacity = d->capacity; a.separate_v = d->separate_v ? 1 : 0;
  a.n_sel = n_sel; a.splits = p.splits; a.rows_per_split = p.rows_per_split; a.sm_scale = sm_scale;
  a.tile_rows = p.tile_rows; a.tiles_per_split = p.tiles_per_split;
  a.q = q; a.topk = topk;
  a.k_nope = c->k.nope; a.k_scale = c->k.scale; a.k_rope = c->k.rope; a.win_k = span ? span_k : c->win_k;
  a.v_nope = c->v.nope; a.v_scale = c->v.scale; a.v_rope = c->v.rope; a.win_v = span ? span_v : c->win_v;
  a.n_tokens = c->n_tokens; a.status = c->status;
  char* w = static_cast<char*>(ws);
  a.part_o = reinterpret_cast<float*>(w);
  a.part_lse = reinterpret_cast<float*>(w + p.part_bytes);
  a.part_lsev = a.part_lse + static_cast<size_t>(a.B) * H * p.splits;
  a.out = out; a.lse = lse;
  if (p.tc) return launch_attention_tc(a, p.head_groups, static_cast<cudaStream_t>(stream));
  return launch_attention(a, p.head_groups, static_cast<cudaStream_t>(stream));
}

// Scratch of dsv4_hca_decode_static: one array per device, never allocated at run time.
static __device__ __align__(256) unsigned char g_static_scratch[DSV4_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch on the current device, looked up once per
// device (cudaGetSymbolAddress with that device current). Null on failure.
void* static_scratch() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

int index_topk_common(const dsv4_layer_desc* d, const dsv4_cache* c, int T, int32_t Hi, const uint16_t* q_idx,
                      const float* w, int32_t k, int32_t* topk, float* scores, void* ws, size_t ws_bytes,
                      void* stream);

}  // namespace
}  // namespace dsv4

using namespace dsv4;

extern "C" {

int dsv4_compress_append(const dsv4_layer_desc* d, const dsv4_cache* c, int32_t T, const uint16_t* k,
                         const uint16_t* v, const uint16_t* z, const float* b, const uint16_t* u,
                         const uint16_t* zu, const float* bu, void* stream) {
  int e = check_desc(d);
  if (e) return e;
  if (!c || T < 0) return DSV4_ERR_INVALID_ARG;
  if ((e = check_kv_planes(c->k, d))) return e;
  if (d->separate_v && (e = check_kv_planes(c->v, d))) return e;
  DSV4_REQ(c->n_tokens);
  DSV4_REQ(c->status);
  if (d->window) {
    DSV4_REQ(c->win_k);
    if (d->separate_v) DSV4_REQ(c->win_v);
  }
  if (d->ratio > 1) {
    DSV4_REQ(c->pend_k);
    DSV4_REQ(c->pend_z);
    if (d->separate_v) DSV4_REQ(c->pend_v);
    if (d->idx_dim) {
      DSV4_REQ(c->pend_u);
      DSV4_REQ(c->pend_zu);
    }
  }
  if (d->idx_dim) {
    DSV4_REQ(c->idx_codes);
    DSV4_REQ(c->idx_scales);
  }
  if (T == 0) return DSV4_OK;
  DSV4_REQ(k);
  DSV4_REQ(z);
  DSV4_REQ(b);
  if (d->separate_v) DSV4_REQ(v);
  if (d->idx_dim) {
    DSV4_REQ(u);
    DSV4_REQ(zu);
    DSV4_REQ(bu);
  }
  AppendArgs a{};
  a.T = T; a.ratio = d->ratio; a.window = d->window; a.capacity = d->capacity; a.d_nope = d->d_nope;
  a.d_rope = d->d_rope; a.idx_dim = d->idx_dim; a.separate_v = d->separate_v ? 1 : 0;
  a.k = k; a.v = v; a.z = z; a.u = u; a.zu = zu; a.bias = b; a.bias_u = bu;
  a.k_nope = c->k.nope; a.k_scale = c->k.scale; a.k_rope = c->k.rope;
  a.v_nope = c->v.nope; a.v_scale = c->v.scale; a.v_rope = c->v.rope;
  a.idx_codes = c->idx_codes; a.idx_scales = c->idx_scales;
  a.win_k = c->win_k; a.win_v = c->win_v; a.pend_k = c->pend_k; a.pend_v = c->pend_v; a.pend_z = c->pend_z;
  a.pend_u = c->pend_u; a.pend_zu = c->pend_zu; a.n_tokens = c->n_tokens; a.status = c->status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int D = d->d_nope + d->d_rope;
  const PoolShape pk = pool_shape(d->ratio, D);
  const PoolShape pu = pool_shape(d->ratio, d->idx_dim ? d->idx_dim : 8);
  const int team_k = pk.G * pk.cg, team_u = d->idx_dim ? pu.G * pu.cg : 0;
  const int part_k = pool_part_floats(pk, d->separate_v != 0), part_u = d->idx_dim ? pool_part_floats(pu, false) : 0;
  if (T == 1) {
    // one CTA per sequence, as large as the largest pooling team
    int threads = team_k > team_u ? team_k : team_u;
    threads = threads < 256 ? 256 : (threads + 31) / 32 * 32;
    const size_t smem = (4 + (part_k > part_u ? part_k : part_u)) * sizeof(float);
    return launch_pdl(append_one_kernel, dim3(d->batch), dim3(threads), smem, st, a);
  }
  const int blocks = (d->ratio - 1 + T) / d->ratio;
  const int win_rows = T < d->window ? T : d->window;
  const int ctas_w = (win_rows + kWinRowsPerCta - 1) / kWinRowsPerCta;
  if (d->ratio > 8 && !d->idx_dim && D % 64 == 0 && D <= 512) {
    // long blocks: each block's channels split over a cluster of D / 64 CTAs
    const int cs = D / 64;
    a.ctas_k = blocks * cs;
    a.ctas_u = 0;
    PoolShape slice = pk;
    slice.cg = 8;
    const int threads = 64 * pk.G / slice_cpt(pk.G);   // 64 to 256
    const size_t smem = static_cast<size_t>(d->ratio) * 64 * (4 + 2 * (d->separate_v ? 3 : 2)) +
                        pool_part_floats(slice, d->separate_v != 0) * sizeof(float) + 4 * sizeof(uint32_t) +
                        128 * sizeof(float);
    static std::once_flag once;
    set_smem_once(once, pool_cluster_kernel, 200 * 1024);
    const int ctas = a.ctas_k + (ctas_w + cs - 1) / cs * cs;
    if ((e = launch_pdl_cluster(pool_cluster_kernel, dim3(ctas, d->batch), dim3(threads), smem, cs, st, a))) return e;
  } else {
    // teams of up to 512 threads, about 256 threads a CTA (several blocks a CTA for small teams)
    a.bpc_k = team_k >= 256 ? 1 : 256 / team_k;
    a.bpc_u = team_u == 0 ? 1 : (team_u >= 256 ? 1 : 256 / team_u);
    const int thr_k = a.bpc_k * team_k, thr_u = a.bpc_u * team_u;
    const int threads = ((thr_k > thr_u ? thr_k : thr_u) + 31) / 32 * 32;
    a.ctas_k = (blocks + a.bpc_k - 1) / a.bpc_k;
    a.ctas_u = d->idx_dim ? (blocks + a.bpc_u - 1) / a.bpc_u : 0;
    const size_t sk = static_cast<size_t>(a.bpc_k) * (part_k + 2), su = static_cast<size_t>(a.bpc_u) * (part_u + 2);
    const size_t smem = (sk > su ? sk : su) * sizeof(float);
    static std::once_flag once;
    set_smem_once(once, pool_chunk_kernel, 160 * 1024);
    const int ctas = a.ctas_k + a.ctas_u + ctas_w;
    if (ctas > 0 && (e = launch_pdl(pool_chunk_kernel, dim3(ctas, d->batch), dim3(threads), smem, st, a))) return e;
  }
  return launch_pdl(append_tail_kernel, dim3(d->batch), dim3(256), 0, st, a);
}

int dsv4_index_topk(const dsv4_layer_desc* d, const dsv4_cache* c, int32_t Hi, const uint16_t* q_idx,
                    const float* w, int32_t k, int32_t* topk, float* scores, void* ws, size_t ws_bytes,
                    void* stream) {
  return index_topk_common(d, c, 1, Hi, q_idx, w, k, topk, scores, ws, ws_bytes, stream);
}

int dsv4_index_topk_multi(const dsv4_layer_desc* d, const dsv4_cache* c, int32_t T, int32_t Hi,
                          const uint16_t* q_idx, const float* w, int32_t k, int32_t* topk, float* scores, void* ws,
                          size_t ws_bytes, void* stream) {
  return index_topk_common(d, c, T, Hi, q_idx, w, k, topk, scores, ws, ws_bytes, stream);
}

}  // extern "C"

namespace dsv4 {
namespace {
int index_topk_common(const dsv4_layer_desc* d, const dsv4_cache* c, int T, int32_t Hi, const uint16_t* q_idx,
                      const float* w, int32_t k, int32_t* topk, float* scores, void* ws, size_t ws_bytes,
                      void* stream) {
  int e = check_desc(d);
  if (e) return e;
  if (!c) return DSV4_ERR_INVALID_ARG;
  if (d->idx_dim == 0) return DSV4_ERR_INVALID_ARG;
  if (Hi < 1 || k < 1 || T < 1) return DSV4_ERR_INVALID_ARG;
  if (Hi > 128 || k > 2048 || static_cast<int64_t>(d->batch) * T > 65535) return DSV4_ERR_UNSUPPORTED;
  DSV4_REQ(c->idx_codes);
  DSV4_REQ(c->idx_scales);
  DSV4_REQ(c->n_tokens);
  DSV4_REQ(c->status);
  DSV4_REQ(q_idx);
  DSV4_REQ(w);
  DSV4_REQ(topk);
  DSV4_REQ(ws);
  if (scores && !aligned16(scores)) return DSV4_ERR_MISALIGNED;
  if (ws_bytes < index_ws_bytes(d, Hi, k, T)) return DSV4_ERR_WORKSPACE;
  const int N = index_heads_padded(Hi);
  const IndexWs wl = index_ws(d, Hi, k, T);
  char* wp = static_cast<char*>(ws);
  IndexArgs a{};
  a.B = d->batch * T; a.T = T;
  a.Hi = Hi; a.N = N; a.Di = d->idx_dim; a.k = k; a.capacity = d->capacity; a.ratio = d->ratio;
  a.q_idx = q_idx; a.w = w; a.n_tokens = c->n_tokens;
  a.q_codes = reinterpret_cast<uint8_t*>(wp + wl.q_codes);
  a.q_scales = reinterpret_cast<uint8_t*>(wp + wl.q_scales);
  a.scores = scores ? scores : reinterpret_cast<float*>(wp + wl.scores);
  a.topk = topk;
  a.hist1 = reinterpret_cast<uint32_t*>(wp + wl.hist1);
  a.hist2 = reinterpret_cast<uint32_t*>(wp + wl.hist2);
  a.cnt = reinterpret_cast<uint32_t*>(wp + wl.cnt);
  a.above = reinterpret_cast<int32_t*>(wp + wl.above);
  a.cand = reinterpret_cast<uint64_t*>(wp + wl.cand);
  a.status = c->status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((e = launch_pdl(quant_query_fp4_kernel, dim3(a.B * N), dim3(32), 0, st, a))) return e;
  IndexTcArgs t{};
  t.B = a.B; t.T = T; t.N = N; t.Di = a.Di; t.capacity = a.capacity; t.ratio = a.ratio;
  const int tiles = (d->capacity + 127) / 128;
  int per_seq = 2 * sm_count() / a.B;
  if (per_seq < 1) per_seq = 1;
  t.ctas_per_seq = per_seq < tiles ? per_seq : tiles;
  uint32_t need = 2 * N + 3 * 4 * (a.Di / 64);
  uint32_t cols = 32;
  while (cols < need) cols <<= 1;
  t.tmem_cols = cols;
  t.n_tokens = c->n_tokens; t.idx_codes = c->idx_codes; t.idx_scales = c->idx_scales; t.q_scales = a.q_scales;
  t.w = w; t.Hi = Hi;
  t.scores = a.scores; t.hist1 = a.hist1; t.cnt = a.cnt; t.k = k; t.status = c->status;
  if ((e = launch_index_scores_tc(t, c->idx_codes, a.q_codes, st))) return e;
  int sel = (2 * sm_count()) / a.B;
  const int sel_max = (d->capacity + 511) / 512;
  if (sel > sel_max) sel = sel_max;
  if (sel < 1) sel = 1;
  return launch_topk_select(a, sel, sm_count(), st);
}
}  // namespace
}  // namespace dsv4

extern "C" {

int dsv4_csa_decode(const dsv4_layer_desc* d, const dsv4_cache* c, int32_t H, const uint16_t* q, float sm_scale,
                    const int32_t* topk, int32_t k, float* out, float* lse, void* ws, size_t ws_bytes,
                    void* stream) {
  if (k < 0) return DSV4_ERR_INVALID_ARG;
  if (k > 2048) return DSV4_ERR_UNSUPPORTED;
  if (k == 0) return decode_common(d, c, H, q, sm_scale, nullptr, -1, out, lse, ws, ws_bytes, stream);
  if (!topk) return DSV4_ERR_INVALID_ARG;
  if (!aligned16(topk)) return DSV4_ERR_MISALIGNED;
  return decode_common(d, c, H, q, sm_scale, topk, k, out, lse, ws, ws_bytes, stream);
}

int dsv4_hca_decode(const dsv4_layer_desc* d, const dsv4_cache* c, int32_t H, const uint16_t* q, float sm_scale,
                    float* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  return decode_common(d, c, H, q, sm_scale, nullptr, 0, out, lse, ws, ws_bytes, stream);
}

int dsv4_csa_decode_multi(const dsv4_layer_desc* d, const dsv4_cache* c, int32_t T, int32_t H, const uint16_t* q,
                          float sm_scale, const int32_t* topk, int32_t k, const uint16_t* span_k,
                          const uint16_t* span_v, float* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  if (k < 0) return DSV4_ERR_INVALID_ARG;
  if (k > 2048) return DSV4_ERR_UNSUPPORTED;
  if (k == 0)
    return decode_common(d, c, H, q, sm_scale, nullptr, -1, out, lse, ws, ws_bytes, stream, T, span_k, span_v);
  if (!topk) return DSV4_ERR_INVALID_ARG;
  if (!aligned16(topk)) return DSV4_ERR_MISALIGNED;
  return decode_common(d, c, H, q, sm_scale, topk, k, out, lse, ws, ws_bytes, stream, T, span_k, span_v);
}

int dsv4_hca_decode_multi(const dsv4_layer_desc* d, const dsv4_cache* c, int32_t T, int32_t H, const uint16_t* q,
                          float sm_scale, const uint16_t* span_k, const uint16_t* span_v, float* out, float* lse,
                          void* ws, size_t ws_bytes, void* stream) {
  return decode_common(d, c, H, q, sm_scale, nullptr, 0, out, lse, ws, ws_bytes, stream, T, span_k, span_v);
}

size_t dsv4_workspace_size_multi(const dsv4_layer_desc* d, int32_t T, int32_t H, int32_t Hi, int32_t k) {
  if (check_desc(d) || T < 1 || static_cast<int64_t>(d->batch) * T > 65535 || H < 1 || H > 128 || Hi < 0 ||
      Hi > 128 || k < 0 || k > 2048)
    return 0;
  size_t need = attn_plan(d, H, 0, T).ws_bytes;
  const size_t win = attn_plan(d, H, -1, T).ws_bytes;
  if (win > need) need = win;
  if (k > 0) {
    const size_t csa = attn_plan(d, H, k, T).ws_bytes;
    if (csa > need) need = csa;
  }
  if (d->idx_dim && Hi > 0) {
    const size_t idx = index_ws_bytes(d, Hi, k > 0 ? k : 1, T);
    if (idx > need) need = idx;
  }
  return need;
}

int dsv4_hca_decode_static(const dsv4_layer_desc* d, const dsv4_cache* c, int32_t H, const uint16_t* q,
                           float sm_scale, float* out, float* lse, void* stream) {
  int e = check_desc(d);
  if (e) return e;
  if (H < 1) return DSV4_ERR_INVALID_ARG;
  if (H > 128) return DSV4_ERR_UNSUPPORTED;
  const size_t need = attn_plan(d, H, 0).ws_bytes;
  if (need > DSV4_STATIC_SCRATCH_BYTES) return DSV4_ERR_SCRATCH;
  void* ws = static_scratch();
  if (!ws) return DSV4_ERR_CUDA;
  return decode_common(d, c, H, q, sm_scale, nullptr, 0, out, lse, ws, DSV4_STATIC_SCRATCH_BYTES, stream);
}

size_t dsv4_workspace_size(const dsv4_layer_desc* d, int32_t H, int32_t Hi, int32_t k) {
  if (check_desc(d) || H < 1 || H > 128 || Hi < 0 || Hi > 128 || k < 0 || k > 2048) return 0;
  size_t need = attn_plan(d, H, 0).ws_bytes;
  const size_t win = attn_plan(d, H, -1).ws_bytes;
  if (win > need) need = win;
  if (k > 0) {
    const size_t csa = attn_plan(d, H, k).ws_bytes;
    if (csa > need) need = csa;
  }
  if (d->idx_dim && Hi > 0) {
    const size_t idx = index_ws_bytes(d, Hi, k > 0 ? k : 1);
    if (idx > need) need = idx;
  }
  return need;
}

int dsv4_decode_plan(const dsv4_layer_desc* d, int32_t H, int32_t k, int32_t* plan) {
  int e = check_desc(d);
  if (e) return e;
  if (!plan || H < 1 || k < -1) return DSV4_ERR_INVALID_ARG;
  if (H > 128 || k > 2048) return DSV4_ERR_UNSUPPORTED;
  const AttnPlan p = attn_plan(d, H, k > 0 ? k : (k == 0 ? -1 : 0));
  plan[0] = p.tc ? 1 : 0;
  plan[1] = p.splits;
  plan[2] = p.tc ? p.tile_rows : p.rows_per_split;
  plan[3] = p.tc ? p.tiles_per_split : 1;
  plan[4] = p.head_groups;
  plan[5] = sm_count();
  return DSV4_OK;
}

int dsv4_project_streams(const dsv4_layer_desc* d, const dsv4_cache* c, int32_t T, int32_t d_model,
                         const uint16_t* hidden, const uint16_t* weight, float rope_base, uint16_t* x, uint16_t* z,
                         uint16_t* u, uint16_t* zu, void* stream) {
  int e = check_desc(d);
  if (e) return e;
  if (!c || T < 0 || d_model <= 0 || !(rope_base > 1.f)) return DSV4_ERR_INVALID_ARG;
  if (d->separate_v) return DSV4_ERR_UNSUPPORTED;
  const int D = d->d_nope + d->d_rope;
  if (d_model % 64 || d->d_nope % 32 || D % 32 || d->idx_dim % 32 || d->d_rope > 64) return DSV4_ERR_UNSUPPORTED;
  DSV4_REQ(c->n_tokens);
  DSV4_REQ(c->status);
  if (T == 0) return DSV4_OK;
  DSV4_REQ(hidden);
  DSV4_REQ(weight);
  DSV4_REQ(x);
  DSV4_REQ(z);
  if (d->idx_dim) {
    DSV4_REQ(u);
    DSV4_REQ(zu);
  }
  ProjArgs a{};
  a.M = d->batch * T;
  a.N = 2 * D + 2 * d->idx_dim;
  a.K = d_model;
  a.T = T;
  a.d_nope = d->d_nope;
  a.d_rope = d->d_rope;
  a.Di = d->idx_dim;
  a.ur = d->d_rope < d->idx_dim ? d->d_rope : d->idx_dim;
  a.n_tokens = c->n_tokens;
  a.x = x; a.z = z; a.u = u; a.zu = zu;
  a.status = c->status;
  return launch_project(a, hidden, weight, static_cast<double>(rope_base), sm_count(), static_cast<cudaStream_t>(stream));
}

int dsv4_debug_force_timeout(int32_t on) { return attention_force_timeout(on); }

int dsv4_read_status(const dsv4_cache* c, void* stream) {
  if (!c || !c->status) return DSV4_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, c->status, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return DSV4_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DSV4_ERR_CUDA;
  if (cudaMemsetAsync(c->status, 0, sizeof(int32_t), st) != cudaSuccess) return DSV4_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DSV4_ERR_CUDA;
  return h;
}

int dsv4_quantize_kv_rows(const float* y, int64_t rows, int32_t d_nope, int32_t d_rope, uint8_t* nope, float* scale,
                          uint16_t* rope, void* stream) {
  if (rows < 0) return DSV4_ERR_INVALID_ARG;
  if (d_nope < 16 || d_nope > 512 || d_nope % 16 || d_rope < 0 || d_rope > 128 || d_rope % 8)
    return DSV4_ERR_UNSUPPORTED;
  if (rows == 0) return DSV4_OK;
  if (!y || !nope || !scale || (d_rope && !rope)) return DSV4_ERR_INVALID_ARG;
  // natural alignment only: rows are read as floats, codes written in pairs
  if ((reinterpret_cast<uintptr_t>(y) & 3) || (reinterpret_cast<uintptr_t>(nope) & 1) ||
      (reinterpret_cast<uintptr_t>(scale) & 3) || (d_rope && (reinterpret_cast<uintptr_t>(rope) & 1)))
    return DSV4_ERR_MISALIGNED;
  const int64_t blocks = (rows + 7) / 8;
  quant_kv_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      y, rows, d_nope, d_rope, nope, scale, rope);
  return launch_status();
}

int dsv4_quantize_fp4_rows(const float* y, int64_t rows, int32_t cols, uint8_t* codes, uint8_t* scales,
                           void* stream) {
  if (rows < 0) return DSV4_ERR_INVALID_ARG;
  if (cols < 32 || cols % 32 || cols > 4096) return DSV4_ERR_UNSUPPORTED;
  if (rows == 0) return DSV4_OK;
  DSV4_REQ(y);
  if (!codes || !scales) return DSV4_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(codes) & 3) return DSV4_ERR_MISALIGNED;
  const int64_t n = rows * (cols / 16);
  quant_fp4_rows_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      y, rows, cols, codes, scales);
  return launch_status();
}

int dsv4_pool_rows(const uint16_t* x, const uint16_t* z, const float* b, int64_t blocks, int32_t ratio, int32_t dim,
                   float* y, void* stream) {
  if (blocks < 0 || ratio < 1 || dim < 1) return DSV4_ERR_INVALID_ARG;
  if (ratio > 256 || dim % 8 || dim > 4096 || blocks > 0x7FFFFFFF) return DSV4_ERR_UNSUPPORTED;
  if (blocks == 0) return DSV4_OK;
  DSV4_REQ(x);
  DSV4_REQ(z);
  DSV4_REQ(b);
  DSV4_REQ(y);
  const PoolShape ps = pool_shape(ratio, dim);
  const int threads = (ps.G * ps.cg + 31) / 32 * 32;
  pool_rows_kernel<<<static_cast<unsigned>(blocks), threads, pool_part_floats(ps, false) * sizeof(float),
                     static_cast<cudaStream_t>(stream)>>>(x, z, b, ratio, dim, y);
  return launch_status();
}

}  // extern "C"
