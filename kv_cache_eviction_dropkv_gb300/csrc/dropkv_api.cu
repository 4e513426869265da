// Host side of the C ABI (include/dropkv.h): argument validation, the
// workspace plan, TMA descriptor encoding and kernel launches.  Nothing here
// allocates device memory; every buffer comes from the caller.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "dropkv_internal.cuh"

namespace dropkv {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

int nr_for(int R) { return R <= 16 ? 16 : R <= 32 ? 32 : R <= 64 ? 64 : -1; }

// SM count of the current device (cached per device ordinal).
int current_sms(int* dev_out) {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev_out) *dev_out = dev;
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev < 64) cache[dev] = sms;
  return sms;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// K or V viewed as a 3-D tensor (d, n_max, B*Hkv) of bf16, loaded as boxes of
// 64 columns x 128 rows with 128-byte swizzle; reads past d or n_max fill zero.
// A [depth][n_max][d] bf16 tensor (K or V: depth = B * Hkv; every query row:
// depth = B * Hq) as boxes of 64 columns x 128 rows, 128-byte swizzled.
bool encode_rows_map(CUtensorMap* map, const void* base, const Geom& g, int depth) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)g.d, (cuuint64_t)g.n_max, (cuuint64_t)depth};
  cuuint64_t strides[2] = {(cuuint64_t)g.d * 2, (cuuint64_t)g.d * 2 * (cuuint64_t)g.n_max};
  cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_kv_map(CUtensorMap* map, const void* base, const Geom& g) { return encode_rows_map(map, base, g, g.U); }

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

bool make_geom(const dropkv_shape* s, int num_sms, Geom* g) {
  if (!s || !g || num_sms <= 0) return false;
  if (s->B < 1 || s->Hq < 1 || s->Hkv < 1 || s->w < 1 || s->n_max < 1) return false;
  if (s->Hq % s->Hkv != 0) return false;
  if (s->d < 8 || s->d > kDPad || s->d % 8 != 0) return false;
  if (s->w > s->n_max) return false;
  const long long R = (long long)(s->Hq / s->Hkv) * s->w;
  if (R > kMaxR) return false;
  const long long U = (long long)s->B * s->Hkv;
  if (U > 65535) return false;   // grid y limit
  g->B = s->B; g->Hq = s->Hq; g->Hkv = s->Hkv; g->d = s->d; g->n_max = s->n_max; g->w = s->w;
  g->g = s->Hq / s->Hkv;
  g->R = (int)R;
  g->NR = nr_for(g->R);
  g->U = (int)U;
  g->tiles_max = ceil_div_i(s->n_max, kTile);
  // One CTA per SM, all resident in a single wave.  With one length for all
  // units each KV head gets floor(SMs / U) CTAs (a CTA more per head would
  // push some into a second wave).  With ragged lengths the kernels share a
  // 1-D grid out over the heads in proportion to their sequences' lengths
  // (read on the device): a head of a sequence twice the mean length can get
  // up to twice its even share of pass-1 partial slots.  The kernels' share
  // arithmetic stays in 32 bits with a grid below 256 CTAs whenever it has
  // more CTAs than units.
  g->ctas = (g->U >= std::min(num_sms, 256)) ? g->U : std::min(num_sms, 256);
  const int per_unit = g->ctas / g->U;
  g->even = std::min(std::min(kMaxSplits, g->tiles_max), per_unit);
  g->splits1 = (g->B == 1) ? g->even : std::max(g->even, std::min(std::min(kMaxSplits, g->tiles_max), 2 * per_unit));
  g->splits2 = g->tiles_max;
  g->chunks = ceil_div_i(s->n_max, kSelChunk);
  g->layer_chunks = ceil_div_i(s->n_max, kLayerChunk);
  return g->NR > 0;
}

WsPlan make_plan(const Geom& g) {
  WsPlan w;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  const size_t UR = (size_t)g.U * g.R;
  w.m = take(UR * 4);          // exported log-sum-exp
  w.a = take(UR * g.d * 4);     // exported attention output
  w.l = take(UR * 4);
  w.m2 = take(UR * 4);
  w.aa = take(UR * 4);
  w.ahl = take((size_t)g.U * 2 * kMaxR * kDPad * 2);
  w.cvec = take((size_t)g.U * kDPad * 4);
  w.cflag = take((size_t)g.U * 4);
  w.dom_s = take(UR * 4);
  w.dom_l = take(UR * 4);
  w.dom_o = take(UR * g.d * 4);
  w.part_o = take((size_t)g.U * g.splits1 * g.R * g.d * 4);
  w.part_ml = take((size_t)g.U * g.splits1 * g.R * 4 * 4);
  w.tile_ctr = take((size_t)g.U * 4);
  w.qwin = take((size_t)g.B * g.Hq * g.w * g.d * 2);
  w.raw = take((size_t)g.U * g.n_max * 4);
  w.sel_zero_begin = off;
  w.hist = take((size_t)g.U * kHistBins * 4);
  w.hist2 = take((size_t)g.U * kHistBins * 4);
  w.cand_cnt = take((size_t)g.U * 4);
  w.sel_tickets = take((size_t)g.U * 2 * 4);
  w.chunk_kept = take((size_t)g.U * g.chunks * 4);
  w.sel_zero_end = off;
  w.sel_state = take((size_t)g.U * 8 * 4);
  w.cand = take((size_t)g.U * kCandCap * 2 * 4);
  w.chunk_off = take((size_t)g.U * g.chunks * 4);
  w.layer_zero_begin = off;
  w.layer_h1 = take((size_t)g.B * kHistBins * 4);
  w.layer_h2 = take((size_t)g.B * kHistBins * 4);
  w.layer_h3 = take((size_t)g.B * 256 * 4);
  w.layer_zero_end = off;
  w.layer_state = take((size_t)g.B * 8 * 4);
  w.layer_counts = take((size_t)g.U * g.layer_chunks * 2 * 4);
  w.total = off;
  return w;
}

}  // namespace dropkv

using namespace dropkv;

extern "C" {

size_t dropkv_workspace_size(const dropkv_shape* shape) {
  const int sms = current_sms(nullptr);
  Geom g;
  if (!make_geom(shape, sms, &g)) return 0;
  return make_plan(g).total;
}

}  // extern "C"

namespace dropkv {

dropkv_status score_core(const dropkv_shape* shape, const void* q_window, const void* k, const void* v,
                         const int32_t* lengths, int32_t pool_kernel, int32_t protect, float* scores,
                         float* raw_scores, void* workspace, size_t workspace_bytes, uint32_t* status,
                         cudaStream_t stream, cudaEvent_t* ev, PoolParams* defer_pool, int kind,
                         bool scoring_regions_only, const PrefillIn* pre) {
  const int sms = current_sms(nullptr);
  if (sms <= 0) return DROPKV_ERR_CUDA;
  if (!shape) return DROPKV_ERR_INVALID_ARG;
  Geom g;
  if (!make_geom(shape, sms, &g)) {
    const bool basic = shape->B >= 1 && shape->Hq >= 1 && shape->Hkv >= 1 && shape->Hq % shape->Hkv == 0 &&
                       shape->w >= 1 && shape->n_max >= shape->w && shape->d >= 1;
    return basic ? DROPKV_ERR_UNSUPPORTED : DROPKV_ERR_INVALID_ARG;
  }
  if (!q_window || !k || !v || !scores || !status) return DROPKV_ERR_INVALID_ARG;
  if (!aligned16(q_window) || !aligned16(k) || !aligned16(v) || !aligned16(scores) ||
      (raw_scores && !aligned16(raw_scores)) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return DROPKV_ERR_INVALID_ARG;
  if (pool_kernel < 1 || pool_kernel > kMaxPool || pool_kernel % 2 == 0 || protect < 0)
    return DROPKV_ERR_INVALID_ARG;
  if (kind != DROPKV_SCORE_DROPKV && kind != DROPKV_SCORE_SNAPKV) return DROPKV_ERR_INVALID_ARG;
  const WsPlan w = make_plan(g);
  // the scoring regions lie ahead of the selection regions
  const size_t need = scoring_regions_only ? w.sel_zero_begin : w.total;
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DROPKV_ERR_WORKSPACE;
  const size_t score_bytes = (size_t)g.U * g.n_max * 4;
  if (raw_scores && ranges_overlap(raw_scores, score_bytes, scores, score_bytes)) return DROPKV_ERR_INVALID_ARG;

  if (pre) {
    // every query row in, the attention output out: [B][Hq][n_max][d] bf16 each
    const size_t rows_bytes = (size_t)g.B * g.Hq * g.n_max * g.d * 2;
    if (!pre->q || !pre->out || !aligned16(pre->q) || !aligned16(pre->out)) return DROPKV_ERR_INVALID_ARG;
    if (ranges_overlap(pre->out, rows_bytes, pre->q, rows_bytes) ||
        ranges_overlap(pre->out, rows_bytes, k, (size_t)g.U * g.n_max * g.d * 2) ||
        ranges_overlap(pre->out, rows_bytes, v, (size_t)g.U * g.n_max * g.d * 2))
      return DROPKV_ERR_INVALID_ARG;
  }

  CUtensorMap tk, tv;
  if (!encode_kv_map(&tk, k, g) || !encode_kv_map(&tv, v, g)) return DROPKV_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q_window);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.lengths = lengths;
  p.B = g.B; p.Hq = g.Hq; p.Hkv = g.Hkv; p.d = g.d; p.n_max = g.n_max; p.w = g.w;
  p.g = g.g; p.R = g.R; p.U = g.U; p.NR = g.NR;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)g.d));
  p.m = reinterpret_cast<float*>(ws + w.m);
  p.l = reinterpret_cast<float*>(ws + w.l);
  p.a = reinterpret_cast<float*>(ws + w.a);
  p.m2 = reinterpret_cast<float*>(ws + w.m2);
  p.aa = reinterpret_cast<float*>(ws + w.aa);
  p.ahl = reinterpret_cast<__nv_bfloat16*>(ws + w.ahl);
  p.cvec = reinterpret_cast<float*>(ws + w.cvec);
  p.cflag = reinterpret_cast<int*>(ws + w.cflag);
  p.dom_s = reinterpret_cast<int*>(ws + w.dom_s);
  p.dom_l = reinterpret_cast<float*>(ws + w.dom_l);
  p.dom_o = reinterpret_cast<float*>(ws + w.dom_o);
  p.part_o = reinterpret_cast<float*>(ws + w.part_o);
  p.part_ml = reinterpret_cast<float*>(ws + w.part_ml);
  p.tile_ctr = reinterpret_cast<uint32_t*>(ws + w.tile_ctr);
  p.raw = raw_scores ? raw_scores : reinterpret_cast<float*>(ws + w.raw);
  p.status = status;
  p.kind = kind == DROPKV_SCORE_SNAPKV ? kKindSnapKV : kKindDropKV;

  if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  p.ctas = g.ctas;
  p.even = (g.B == 1 || !lengths) ? g.even : 0;
  p.splits = g.splits1;
  p.splits1 = g.splits1;
  if (pre) {
    // the prefill attention takes pass 1's place: one partial state per window row
    CUtensorMap tq;
    if (!encode_rows_map(&tq, pre->q, g, g.B * g.Hq)) return DROPKV_ERR_CUDA;
    PrefillParams pf{};
    pf.q = static_cast<const __nv_bfloat16*>(pre->q);
    pf.out = static_cast<__nv_bfloat16*>(pre->out);
    pf.q_win = reinterpret_cast<__nv_bfloat16*>(ws + w.qwin);
    pf.lengths = lengths;
    pf.part_o = p.part_o;
    pf.part_ml = p.part_ml;
    pf.B = g.B; pf.Hq = g.Hq; pf.Hkv = g.Hkv; pf.g = g.g; pf.d = g.d; pf.n_max = g.n_max; pf.w = g.w;
    pf.R = g.R; pf.splits = g.splits1;
    pf.scale_log2 = p.scale_log2;
    pf.status = status;
    if (launch_prefill(pf, tq, tk, tv, stream) != cudaSuccess) return DROPKV_ERR_CUDA;
    p.q = pf.q_win;
    p.part_splits = 1;
  } else if (launch_window_attention(p, g.NR, tk, tv, g.splits1, stream) != cudaSuccess) {
    return DROPKV_ERR_CUDA;
  }
  if (ev && cudaEventRecord(ev[1], stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  if (launch_merge(p, stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  if (ev && cudaEventRecord(ev[2], stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  p.splits = g.splits2;
  if (launch_score(p, g.NR, tk, tv, stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  if (ev && cudaEventRecord(ev[3], stream) != cudaSuccess) return DROPKV_ERR_CUDA;

  PoolParams pp{};
  pp.raw = p.raw;
  pp.scores = scores;
  pp.lengths = lengths;
  pp.B = g.B; pp.Hkv = g.Hkv; pp.n_max = g.n_max; pp.w = g.w;
  pp.half = pool_kernel / 2;
  pp.protect = protect;
  pp.status = status;
  if (defer_pool) {   // the caller's selection pools (dropkv_evict)
    *defer_pool = pp;
    return DROPKV_OK;
  }
  if (launch_pool_protect(pp, stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  if (ev && cudaEventRecord(ev[4], stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  return DROPKV_OK;
}

}  // namespace dropkv

namespace {

dropkv_status score_impl(const dropkv_shape* shape, const void* q_window, const void* k, const void* v,
                         const int32_t* lengths, int32_t pool_kernel, int32_t protect, float* scores,
                         float* raw_scores, void* workspace, size_t workspace_bytes, uint32_t* status,
                         cudaStream_t stream, cudaEvent_t* ev, PoolParams* defer_pool = nullptr,
                         int kind = DROPKV_SCORE_DROPKV, const PrefillIn* pre = nullptr) {
  return score_core(shape, q_window, k, v, lengths, pool_kernel, protect, scores, raw_scores, workspace,
                    workspace_bytes, status, stream, ev, defer_pool, kind, false, pre);
}

dropkv_status select_impl(const dropkv_shape* shape, const float* scores, const int32_t* lengths,
                          const int32_t* evict_k, int32_t protect, int32_t* kept_idx, int32_t* kept_len,
                          void* workspace, size_t workspace_bytes, uint32_t* status, cudaStream_t stream,
                          const PoolParams* pool, bool check_only = false) {
  const int sms = current_sms(nullptr);
  if (sms <= 0) return DROPKV_ERR_CUDA;
  Geom g;
  if (!shape || !make_geom(shape, sms, &g)) return DROPKV_ERR_INVALID_ARG;
  if (!scores || !evict_k || !kept_idx || !kept_len || !status || protect < 0) return DROPKV_ERR_INVALID_ARG;
  if (!aligned16(scores) || !aligned16(kept_idx)) return DROPKV_ERR_INVALID_ARG;
  const WsPlan w = make_plan(g);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return DROPKV_ERR_WORKSPACE;
  if (check_only) return DROPKV_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SelParams p{};
  p.scores = scores;
  p.lengths = lengths;
  p.evict_k = evict_k;
  p.kept_idx = kept_idx;
  p.kept_len = kept_len;
  p.B = g.B; p.Hkv = g.Hkv; p.n_max = g.n_max; p.protect = protect; p.chunks = g.chunks;
  p.hist = reinterpret_cast<uint32_t*>(ws + w.hist);
  p.hist2 = reinterpret_cast<uint32_t*>(ws + w.hist2);
  p.state = reinterpret_cast<uint32_t*>(ws + w.sel_state);
  p.cand = reinterpret_cast<uint32_t*>(ws + w.cand);
  p.cand_cnt = reinterpret_cast<uint32_t*>(ws + w.cand_cnt);
  p.tickets = reinterpret_cast<uint32_t*>(ws + w.sel_tickets);
  p.chunk_kept = reinterpret_cast<uint32_t*>(ws + w.chunk_kept);
  p.chunk_off = reinterpret_cast<uint32_t*>(ws + w.chunk_off);
  p.status = status;
  if (pool) p.pool = *pool;
  return launch_select(p, w.sel_zero_end - w.sel_zero_begin, ws + w.sel_zero_begin, stream) == cudaSuccess
             ? DROPKV_OK
             : DROPKV_ERR_CUDA;
}

dropkv_status compact_impl(const dropkv_shape* shape, const void* k, const void* v, const int32_t* kept_idx,
                           const int32_t* kept_len, int32_t out_rows, void* k_out, void* v_out, uint32_t* status,
                           cudaStream_t stream, bool check_only, bool per_head = false) {
  const int sms = current_sms(nullptr);
  if (sms <= 0) return DROPKV_ERR_CUDA;
  Geom g;
  if (!shape || !make_geom(shape, sms, &g)) return DROPKV_ERR_INVALID_ARG;
  if (!k || !v || !kept_idx || !kept_len || !k_out || !v_out || !status || out_rows < 0)
    return DROPKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out)) return DROPKV_ERR_INVALID_ARG;
  const size_t in_bytes = (size_t)g.U * g.n_max * g.d * 2, out_bytes = (size_t)g.U * out_rows * g.d * 2;
  if (out_rows > 0 && (ranges_overlap(k_out, out_bytes, k, in_bytes) || ranges_overlap(k_out, out_bytes, v, in_bytes) ||
                       ranges_overlap(v_out, out_bytes, k, in_bytes) || ranges_overlap(v_out, out_bytes, v, in_bytes) ||
                       ranges_overlap(k_out, out_bytes, v_out, out_bytes)))
    return DROPKV_ERR_INVALID_ARG;
  if (check_only) return DROPKV_OK;
  CompactParams p{};
  p.k = static_cast<const uint8_t*>(k);
  p.v = static_cast<const uint8_t*>(v);
  p.kept_idx = kept_idx;
  p.kept_len = kept_len;
  p.k_out = static_cast<uint8_t*>(k_out);
  p.v_out = static_cast<uint8_t*>(v_out);
  p.B = g.B; p.Hkv = g.Hkv; p.n_max = g.n_max; p.row_bytes = g.d * 2; p.out_rows = out_rows;
  p.status = status;
  p.per_head = per_head ? 1 : 0;
  return launch_compact(p, stream) == cudaSuccess ? DROPKV_OK : DROPKV_ERR_CUDA;
}

}  // namespace

extern "C" {

dropkv_status dropkv_score(const dropkv_shape* shape, const void* q_window, const void* k, const void* v,
                           const int32_t* lengths, int32_t pool_kernel, int32_t protect, float* scores,
                           float* raw_scores, void* workspace, size_t workspace_bytes, uint32_t* status,
                           cudaStream_t stream) {
  return score_impl(shape, q_window, k, v, lengths, pool_kernel, protect, scores, raw_scores, workspace,
                    workspace_bytes, status, stream, nullptr);
}

dropkv_status dropkv_score_timed(const dropkv_shape* shape, int32_t score_kind, const void* q_window, const void* k,
                                 const void* v, const int32_t* lengths, int32_t pool_kernel, int32_t protect,
                                 float* scores, float* raw_scores, void* workspace, size_t workspace_bytes,
                                 uint32_t* status, cudaStream_t stream, cudaEvent_t* phase_events) {
  if (!phase_events) return DROPKV_ERR_INVALID_ARG;
  return score_impl(shape, q_window, k, v, lengths, pool_kernel, protect, scores, raw_scores, workspace,
                    workspace_bytes, status, stream, phase_events, nullptr, score_kind);
}

dropkv_status dropkv_select(const dropkv_shape* shape, const float* scores, const int32_t* lengths,
                            const int32_t* evict_k, int32_t protect, int32_t* kept_idx, int32_t* kept_len,
                            void* workspace, size_t workspace_bytes, uint32_t* status, cudaStream_t stream) {
  return select_impl(shape, scores, lengths, evict_k, protect, kept_idx, kept_len, workspace, workspace_bytes, status,
                     stream, nullptr);
}

dropkv_status dropkv_compact(const dropkv_shape* shape, const void* k, const void* v, const int32_t* kept_idx,
                             const int32_t* kept_len, int32_t out_rows, void* k_out, void* v_out,
                             uint32_t* status, cudaStream_t stream) {
  return compact_impl(shape, k, v, kept_idx, kept_len, out_rows, k_out, v_out, status, stream, false);
}

}  // extern "C"

namespace {

// Score, select and compact in one call (dropkv_evict_ex, and with `pre` the
// prefilled variant).
dropkv_status evict_core(const dropkv_shape* shape, int32_t score_kind, const void* q_window, const void* k,
                         const void* v, const int32_t* lengths, const int32_t* evict_k, int32_t pool_kernel,
                         int32_t protect, float* scores, float* raw_scores, int32_t* kept_idx, int32_t* kept_len,
                         int32_t out_rows, void* k_out, void* v_out, void* workspace, size_t workspace_bytes,
                         uint32_t* status, cudaStream_t stream, const PrefillIn* pre) {
  // every argument is checked before anything is launched
  dropkv_status st = select_impl(shape, scores, lengths, evict_k, protect, kept_idx, kept_len, workspace,
                                 workspace_bytes, status, stream, nullptr, /*check_only=*/true);
  if (st != DROPKV_OK) return st;
  if ((k_out == nullptr) != (v_out == nullptr)) return DROPKV_ERR_INVALID_ARG;
  if (k_out) {
    st = compact_impl(shape, k, v, kept_idx, kept_len, out_rows, k_out, v_out, status, stream, true);
    if (st != DROPKV_OK) return st;
  }
  PoolParams pool{};
  st = score_impl(shape, q_window, k, v, lengths, pool_kernel, protect, scores, raw_scores, workspace,
                  workspace_bytes, status, stream, nullptr, &pool, score_kind, pre);
  if (st != DROPKV_OK) return st;
  st = select_impl(shape, scores, lengths, evict_k, protect, kept_idx, kept_len, workspace, workspace_bytes, status,
                   stream, &pool);
  if (st != DROPKV_OK || !k_out) return st;
  return compact_impl(shape, k, v, kept_idx, kept_len, out_rows, k_out, v_out, status, stream, false);
}

}  // namespace

extern "C" {

dropkv_status dropkv_evict_ex(const dropkv_shape* shape, int32_t score_kind, const void* q_window, const void* k,
                              const void* v, const int32_t* lengths, const int32_t* evict_k, int32_t pool_kernel,
                              int32_t protect, float* scores, float* raw_scores, int32_t* kept_idx,
                              int32_t* kept_len, int32_t out_rows, void* k_out, void* v_out, void* workspace,
                              size_t workspace_bytes, uint32_t* status, cudaStream_t stream) {
  return evict_core(shape, score_kind, q_window, k, v, lengths, evict_k, pool_kernel, protect, scores, raw_scores,
                    kept_idx, kept_len, out_rows, k_out, v_out, workspace, workspace_bytes, status, stream, nullptr);
}

dropkv_status dropkv_prefill_attention(const dropkv_shape* shape, const void* q, const void* k, const void* v,
                                       const int32_t* lengths, void* attn_out, void* workspace,
                                       size_t workspace_bytes, uint32_t* status, cudaStream_t stream) {
  const int sms = current_sms(nullptr);
  if (sms <= 0) return DROPKV_ERR_CUDA;
  Geom g;
  if (!shape || !make_geom(shape, sms, &g)) return DROPKV_ERR_INVALID_ARG;
  if (!q || !k || !v || !attn_out || !status) return DROPKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(attn_out) ||
      (reinterpret_cast<uintptr_t>(status) & 3u))
    return DROPKV_ERR_INVALID_ARG;
  const size_t rows_bytes = (size_t)g.B * g.Hq * g.n_max * g.d * 2;
  const size_t kv_bytes = (size_t)g.U * g.n_max * g.d * 2;
  if (ranges_overlap(attn_out, rows_bytes, q, rows_bytes) || ranges_overlap(attn_out, rows_bytes, k, kv_bytes) ||
      ranges_overlap(attn_out, rows_bytes, v, kv_bytes))
    return DROPKV_ERR_INVALID_ARG;
  const WsPlan w = make_plan(g);
  if (!workspace || workspace_bytes < w.sel_zero_begin || !aligned16(workspace)) return DROPKV_ERR_WORKSPACE;
  CUtensorMap tq, tk, tv;
  if (!encode_rows_map(&tq, q, g, g.B * g.Hq) || !encode_kv_map(&tk, k, g) || !encode_kv_map(&tv, v, g))
    return DROPKV_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PrefillParams pf{};
  pf.q = static_cast<const __nv_bfloat16*>(q);
  pf.out = static_cast<__nv_bfloat16*>(attn_out);
  pf.q_win = reinterpret_cast<__nv_bfloat16*>(ws + w.qwin);
  pf.lengths = lengths;
  pf.part_o = reinterpret_cast<float*>(ws + w.part_o);
  pf.part_ml = reinterpret_cast<float*>(ws + w.part_ml);
  pf.B = g.B; pf.Hq = g.Hq; pf.Hkv = g.Hkv; pf.g = g.g; pf.d = g.d; pf.n_max = g.n_max; pf.w = g.w;
  pf.R = g.R; pf.splits = g.splits1;
  pf.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)g.d));
  pf.status = status;
  return launch_prefill(pf, tq, tk, tv, stream) == cudaSuccess ? DROPKV_OK : DROPKV_ERR_CUDA;
}

dropkv_status dropkv_evict_prefill(const dropkv_shape* shape, int32_t score_kind, const void* q, const void* k,
                                   const void* v, const int32_t* lengths, const int32_t* evict_k,
                                   int32_t pool_kernel, int32_t protect, void* attn_out, float* scores,
                                   float* raw_scores, int32_t* kept_idx, int32_t* kept_len, int32_t out_rows,
                                   void* k_out, void* v_out, void* workspace, size_t workspace_bytes,
                                   uint32_t* status, cudaStream_t stream) {
  const PrefillIn pre{q, attn_out};
  // q stands in for the window argument in the argument checks; pass 2 reads
  // the window rows the prefill kernel copies into the workspace
  return evict_core(shape, score_kind, q, k, v, lengths, evict_k, pool_kernel, protect, scores, raw_scores, kept_idx,
                    kept_len, out_rows, k_out, v_out, workspace, workspace_bytes, status, stream, &pre);
}

dropkv_status dropkv_evict(const dropkv_shape* shape, const void* q_window, const void* k, const void* v,
                           const int32_t* lengths, const int32_t* evict_k, int32_t pool_kernel, int32_t protect,
                           float* scores, float* raw_scores, int32_t* kept_idx, int32_t* kept_len, int32_t out_rows,
                           void* k_out, void* v_out, void* workspace, size_t workspace_bytes, uint32_t* status,
                           cudaStream_t stream) {
  return dropkv_evict_ex(shape, DROPKV_SCORE_DROPKV, q_window, k, v, lengths, evict_k, pool_kernel, protect, scores,
                         raw_scores, kept_idx, kept_len, out_rows, k_out, v_out, workspace, workspace_bytes, status,
                         stream);
}

dropkv_status dropkv_score_ex(const dropkv_shape* shape, int32_t score_kind, const void* q_window, const void* k,
                              const void* v, const int32_t* lengths, int32_t pool_kernel, int32_t protect,
                              float* scores, float* raw_scores, void* workspace, size_t workspace_bytes,
                              uint32_t* status, cudaStream_t stream) {
  return score_impl(shape, q_window, k, v, lengths, pool_kernel, protect, scores, raw_scores, workspace,
                    workspace_bytes, status, stream, nullptr, nullptr, score_kind);
}

dropkv_status dropkv_select_layer(const dropkv_shape* shape, const float* scores, const int32_t* lengths,
                                  const int32_t* evict_total, int32_t protect, int32_t* kept_idx, int32_t* kept_len,
                                  void* workspace, size_t workspace_bytes, uint32_t* status, cudaStream_t stream) {
  const int sms = current_sms(nullptr);
  if (sms <= 0) return DROPKV_ERR_CUDA;
  Geom g;
  if (!shape || !make_geom(shape, sms, &g)) return DROPKV_ERR_INVALID_ARG;
  if (!scores || !evict_total || !kept_idx || !kept_len || !status || protect < 0) return DROPKV_ERR_INVALID_ARG;
  if (!aligned16(scores) || !aligned16(kept_idx)) return DROPKV_ERR_INVALID_ARG;
  if ((long long)g.Hkv * g.n_max >= (1LL << 31)) return DROPKV_ERR_UNSUPPORTED;
  const WsPlan w = make_plan(g);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return DROPKV_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  LayerSelParams p{};
  p.scores = scores;
  p.lengths = lengths;
  p.evict_total = evict_total;
  p.kept_idx = kept_idx;
  p.kept_len = kept_len;
  p.B = g.B; p.Hkv = g.Hkv; p.n_max = g.n_max; p.protect = protect; p.chunks = g.layer_chunks;
  p.h1 = reinterpret_cast<uint32_t*>(ws + w.layer_h1);
  p.h2 = reinterpret_cast<uint32_t*>(ws + w.layer_h2);
  p.h3 = reinterpret_cast<uint32_t*>(ws + w.layer_h3);
  p.state = reinterpret_cast<uint32_t*>(ws + w.layer_state);
  p.counts = reinterpret_cast<uint32_t*>(ws + w.layer_counts);
  p.status = status;
  return launch_select_layer(p, w.layer_zero_end - w.layer_zero_begin, ws + w.layer_zero_begin, stream) ==
                 cudaSuccess
             ? DROPKV_OK
             : DROPKV_ERR_CUDA;
}

dropkv_status dropkv_compact_heads(const dropkv_shape* shape, const void* k, const void* v, const int32_t* kept_idx,
                                   const int32_t* kept_len, int32_t out_rows, void* k_out, void* v_out,
                                   uint32_t* status, cudaStream_t stream) {
  return compact_impl(shape, k, v, kept_idx, kept_len, out_rows, k_out, v_out, status, stream, false, true);
}

dropkv_status dropkv_read_status(const uint32_t* status, cudaStream_t stream, uint32_t* flags_out) {
  if (!status) return DROPKV_ERR_INVALID_ARG;
  uint32_t f = 0;
  if (cudaMemcpyAsync(&f, status, sizeof f, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  if (flags_out) *flags_out = f;
  if (f & DROPKV_FLAG_SINGULAR) return DROPKV_ERR_SINGULAR;
  if (f & DROPKV_FLAG_NONFINITE) return DROPKV_ERR_NONFINITE;
  if (f & (DROPKV_FLAG_BAD_LENGTH | DROPKV_FLAG_BAD_K | DROPKV_FLAG_OVERFLOW)) return DROPKV_ERR_DEVICE_ARG;
  if (f & DROPKV_FLAG_TIMEOUT) return DROPKV_ERR_TIMEOUT;
  if (f & DROPKV_FLAG_INTERNAL) return DROPKV_ERR_CUDA;
  return DROPKV_OK;
}

const char* dropkv_version(void) { return "dropkv-gb300 0.1 (sm_103a, tcgen05/TMA)"; }

}  // extern "C"
