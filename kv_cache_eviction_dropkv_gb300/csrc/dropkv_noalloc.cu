// dropkv_score_noalloc: dropkv_score for callers that cannot allocate device
// memory when they score -- for example a host framework that owns all device
// memory through its own pool and gives this library no allocator, or a
// serving loop that forbids allocations after start-up so that a step can
// never stall in, or fail on, cudaMalloc.  The caller still owns inputs and
// outputs; only the scratch moves into a fixed device array of this file.
#include <cuda_runtime.h>

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

}  // namespace
}  // namespace dropkv

using namespace dropkv;

// The same scoring as dropkv_score, with the array as its workspace: shapes
// whose scoring regions exceed the array get DROPKV_ERR_WORKSPACE from the
// shared argument checks, and nothing is launched.  The array keeps the
// previous call's contents; scoring writes every scratch value before reading
// it (the merge kernel resets pass 2's tile counters), so nothing has to be
// cleared first.
extern "C" dropkv_status dropkv_score_noalloc(const dropkv_shape* shape, const void* q_window, const void* k,
                                              const void* v, const int32_t* lengths, int32_t pool_kernel,
                                              int32_t protect, float* scores, float* raw_scores, uint32_t* status,
                                              cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DROPKV_ERR_CUDA;
  void* ws = scratch_address(dev);
  if (!ws) return DROPKV_ERR_CUDA;
  return score_core(shape, q_window, k, v, lengths, pool_kernel, protect, scores, raw_scores, ws,
                    kNoAllocScratchBytes, status, stream, nullptr, nullptr, DROPKV_SCORE_DROPKV,
                    /*scoring_regions_only=*/true);
}
