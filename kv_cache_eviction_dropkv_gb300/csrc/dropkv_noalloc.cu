// dropkv_score_noalloc: dropkv_score for callers that cannot allocate device
// memory when they score -- for example a host framework that owns all device
// memory through its own pool and gives this library no allocator, or a
// serving loop that forbids allocations after start-up so that a step can
// never stall in, or fail on, cudaMalloc.  The caller still owns inputs and
// outputs; only the scratch moves into a fixed device array of this file.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "dropkv_internal.cuh"

namespace dropkv {
namespace {

// Scratch of the allocation-free call.  Every GPU that loads the library
// holds it until the process exits; every call shares it.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of the scratch array for `dev` (the current device).  Host
// code may not use the symbol itself: in host code it is only a stand-in.
void* scratch_address(int dev) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 noalloc_encoder() {
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

bool noalloc_kv_map(CUtensorMap* map, const void* base, const Geom& g) {
  auto enc = noalloc_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)g.d, (cuuint64_t)g.n_max, (cuuint64_t)g.U};
  cuuint64_t strides[2] = {(cuuint64_t)g.d * 2, (cuuint64_t)g.d * 2 * (cuuint64_t)g.n_max};
  cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dropkv

using namespace dropkv;

extern "C" dropkv_status dropkv_score_noalloc(const dropkv_shape* shape, const void* q_window, const void* k,
                                              const void* v, const int32_t* lengths, int32_t pool_kernel,
                                              int32_t protect, float* scores, float* raw_scores, uint32_t* status,
                                              cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DROPKV_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DROPKV_ERR_CUDA;
  if (!shape) return DROPKV_ERR_INVALID_ARG;
  Geom g;
  if (!make_geom(shape, sms, &g)) {
    const bool basic = shape->B >= 1 && shape->Hq >= 1 && shape->Hkv >= 1 && shape->Hq % shape->Hkv == 0 &&
                       shape->w >= 1 && shape->n_max >= shape->w && shape->d >= 1;
    return basic ? DROPKV_ERR_UNSUPPORTED : DROPKV_ERR_INVALID_ARG;
  }
  if (!q_window || !k || !v || !scores || !status) return DROPKV_ERR_INVALID_ARG;
  if (!is_aligned16(q_window) || !is_aligned16(k) || !is_aligned16(v) || !is_aligned16(scores) ||
      (raw_scores && !is_aligned16(raw_scores)) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return DROPKV_ERR_INVALID_ARG;
  if (pool_kernel < 1 || pool_kernel > kMaxPool || pool_kernel % 2 == 0 || protect < 0)
    return DROPKV_ERR_INVALID_ARG;
  const WsPlan w = make_plan(g);
  // the scoring regions are the ones ahead of the selection regions
  if (w.sel_zero_begin > kNoAllocScratchBytes) return DROPKV_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(scratch_address(dev));
  if (!ws) return DROPKV_ERR_CUDA;

  CUtensorMap tk, tv;
  if (!noalloc_kv_map(&tk, k, g) || !noalloc_kv_map(&tv, v, g)) return DROPKV_ERR_CUDA;
  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q_window);
  p.lengths = lengths;
  p.B = g.B; p.Hq = g.Hq; p.Hkv = g.Hkv; p.d = g.d; p.n_max = g.n_max; p.w = g.w;
  p.g = g.g; p.R = g.R; p.U = g.U;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)g.d));
  p.m = reinterpret_cast<float*>(ws + w.m);
  p.l = reinterpret_cast<float*>(ws + w.l);
  p.a = reinterpret_cast<float*>(ws + w.a);
  p.m2 = reinterpret_cast<float*>(ws + w.m2);
  p.aa = reinterpret_cast<float*>(ws + w.aa);
  p.ahl = reinterpret_cast<__nv_bfloat16*>(ws + w.ahl);
  p.part_o = reinterpret_cast<float*>(ws + w.part_o);
  p.part_ml = reinterpret_cast<float*>(ws + w.part_ml);
  p.tile_ctr = reinterpret_cast<uint32_t*>(ws + w.tile_ctr);
  p.raw = raw_scores ? raw_scores : reinterpret_cast<float*>(ws + w.raw);
  p.status = status;
  // the array keeps the previous call's contents; scoring writes every scratch
  // value before reading it (the merge kernel resets pass 2's tile counters),
  // so nothing has to be cleared first
  p.ctas = g.ctas;
  p.even = (g.B == 1 || !lengths) ? g.even : 0;
  p.splits = g.splits1;
  if (launch_window_attention(p, g.NR, tk, tv, g.splits1, stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  if (launch_merge(p, stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  p.splits = g.splits2;
  if (launch_score(p, g.NR, tk, tv, stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  PoolParams pp{};
  pp.raw = p.raw;
  pp.scores = scores;
  pp.lengths = lengths;
  pp.B = g.B; pp.Hkv = g.Hkv; pp.n_max = g.n_max; pp.w = g.w;
  pp.half = pool_kernel / 2;
  pp.protect = protect;
  pp.status = status;
  if (launch_pool_protect(pp, stream) != cudaSuccess) return DROPKV_ERR_CUDA;
  return DROPKV_OK;
}
