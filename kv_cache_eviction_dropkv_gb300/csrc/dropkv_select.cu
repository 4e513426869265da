// Pool + protect, bottom-k selection and compaction of the DropKV path.
//
// "DropKV: Exact single-entry output-perturbation scoring", Algorithm 1
// summary: MaxPool1D over the sequence, the recent observation window set to
// +inf, then the smallest scores are evicted.  "DropKV: Decoupling ...",
// section 2.2: eviction removes tokens and shrinks the resident cache.
//
// Selection is an exact radix select on the pair (order-preserving key of the
// float score, position): the k-th smallest pair (T, t) splits the evicted
// pairs (<= (T, t)) from the kept ones, so ties on the score go to the lower
// position first and exactly k_b slots are evicted.
//   1. select_hist:  histogram of the top 12 key bits per KV head (all CTAs),
//                    the last CTA of a head locates the bin holding rank k.
//   2. select_cand:  CTAs count the slots above that bin per chunk and gather
//                    the bin's members; the last CTA resolves the remaining
//                    52 bits of (key, position) in shared memory and turns the
//                    per-chunk kept counts into output offsets.
//   3. select_write: each chunk writes its kept positions in ascending order.
#include <cuda_runtime.h>

#include "dropkv_internal.cuh"

namespace dropkv {
namespace {

constexpr int kSelThreads = 256;
constexpr int kPerThread = kSelChunk / kSelThreads;   // 16
constexpr int kPoolTile = 2048;
constexpr int kPoolThreads = 256;

enum : uint32_t { kModeNormal = 0, kModeKeepAll = 1, kModeSkip = 2 };
enum { kStMode = 0, kStBin = 1, kStRank = 2, kStCount = 3, kStKey = 4, kStIdx = 5 };

__device__ __forceinline__ uint32_t f2ord(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Exclusive scan of one value per thread over the block; returns the prefix
// and writes the block total to *total.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* scratch, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = (lane < NT / 32) ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NT / 32) scratch[lane] = s;
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? scratch[warp - 1] : 0u) + x - v;
  *total = scratch[NT / 32 - 1];
  __syncthreads();
  return before;
}

// ------------------------------------------------------------ pool + protect
__global__ void __launch_bounds__(kPoolThreads) pool_protect_kernel(const PoolParams p) {
  __shared__ float buf[kPoolTile + 2 * (kMaxPool / 2)];
  const int unit = blockIdx.y, b = unit / p.Hkv;
  const int nb = p.lengths ? p.lengths[b] : p.n_max;
  if (nb < p.w || nb > p.n_max) return;
  const int j0 = blockIdx.x * kPoolTile;
  if (j0 >= nb) return;
  const float* raw = p.raw + (size_t)unit * p.n_max;
  float* out = p.scores + (size_t)unit * p.n_max;
  const int half = p.half, span = kPoolTile + 2 * half;
  for (int i = threadIdx.x; i < span; i += kPoolThreads) {
    const int jj = j0 - half + i;
    buf[i] = (jj >= 0 && jj < nb) ? raw[jj] : -INFINITY;
  }
  __syncthreads();
  const int first_protected = nb - p.protect;
  for (int i = threadIdx.x; i < kPoolTile; i += kPoolThreads) {
    const int j = j0 + i;
    if (j >= nb) break;
    float m = buf[i];
    for (int t = 1; t <= 2 * half; ++t) m = fmaxf(m, buf[i + t]);
    out[j] = (j >= first_protected) ? INFINITY : m;
  }
}

// ------------------------------------------------------------ selection
struct UnitInfo {
  int nb, kb;
  uint32_t mode;
};

__device__ __forceinline__ UnitInfo unit_info(const SelParams& p, int b) {
  UnitInfo u;
  u.nb = p.lengths ? p.lengths[b] : p.n_max;
  u.kb = p.evict_k[b];
  if (u.nb < 1 || u.nb > p.n_max || u.nb < p.protect) u.mode = kModeSkip;
  else if (u.kb < 0 || u.kb > u.nb - p.protect) u.mode = kModeKeepAll;
  else if (u.kb == 0) u.mode = kModeKeepAll;
  else u.mode = kModeNormal;
  return u;
}

__global__ void __launch_bounds__(kSelThreads) select_hist_kernel(const SelParams p) {
  __shared__ uint32_t sh[kHistBins];
  __shared__ uint32_t scratch[32];
  __shared__ int is_last;
  const int chunk = blockIdx.x, unit = blockIdx.y, b = unit / p.Hkv, h = unit - b * p.Hkv;
  const UnitInfo ui = unit_info(p, b);
  uint32_t* st = p.state + (size_t)unit * 8;
  if (chunk == 0 && h == 0 && threadIdx.x == 0) {
    if (ui.mode == kModeSkip) atomicOr(p.status, DROPKV_FLAG_BAD_LENGTH);
    else if (ui.kb < 0 || ui.kb > ui.nb - p.protect) atomicOr(p.status, DROPKV_FLAG_BAD_K);
  }
  if (ui.mode == kModeSkip) {
    if (chunk == 0 && threadIdx.x == 0) st[kStMode] = kModeSkip;
    return;
  }
  const int j0 = chunk * kSelChunk;
  if (j0 >= ui.nb) return;
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) sh[i] = 0;
  __syncthreads();
  const float* sc = p.scores + (size_t)unit * p.n_max;
  for (int i = 0; i < kPerThread; ++i) {
    const int j = j0 + i * kSelThreads + threadIdx.x;
    if (j < ui.nb) atomicAdd(&sh[f2ord(sc[j]) >> 20], 1u);
  }
  __syncthreads();
  uint32_t* gh = p.hist + (size_t)unit * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t t = atomicAdd(&p.tickets[unit * 2], 1u);
    is_last = (t == (uint32_t)ceil_div(ui.nb, kSelChunk) - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // last CTA of this head: find the bin holding the kb-th smallest key
  uint32_t cnt[kHistBins / kSelThreads];
  uint32_t local = 0;
  for (int q = 0; q < kHistBins / kSelThreads; ++q) {
    cnt[q] = __ldcg(&gh[threadIdx.x * (kHistBins / kSelThreads) + q]);
    local += cnt[q];
  }
  uint32_t total;
  const uint32_t before = block_exclusive_scan<kSelThreads>(local, scratch, &total);
  if (ui.mode == kModeNormal) {
    const uint32_t k = (uint32_t)ui.kb;
    if (before < k && k <= before + local) {
      uint32_t c = before;
      for (int q = 0; q < kHistBins / kSelThreads; ++q) {
        if (c + cnt[q] >= k) {
          st[kStBin] = threadIdx.x * (kHistBins / kSelThreads) + q;
          st[kStRank] = k - c;
          st[kStCount] = cnt[q];
          break;
        }
        c += cnt[q];
      }
    }
  }
  if (threadIdx.x == 0) {
    st[kStMode] = ui.mode;
    p.tickets[unit * 2] = 0;
  }
}

// Radix select of the rank-th (1-based) smallest 64-bit composite among `n`
// items whose top 12 bits are already fixed; `get(i)` returns item i.
// Resolves bits 51..0 with 8-bit digits; returns the selected composite.
template <typename Get>
__device__ uint64_t radix_select_52(int n, uint32_t rank, uint64_t prefix, Get get, uint32_t* hist,
                                    uint32_t* scratch) {
  __shared__ uint64_t s_prefix;
  __shared__ uint32_t s_rank, s_count;
  if (threadIdx.x == 0) { s_prefix = prefix; s_rank = rank; s_count = (uint32_t)n; }
  __syncthreads();
  const int shifts[7] = {44, 36, 28, 20, 12, 4, 0};
  const int widths[7] = {8, 8, 8, 8, 8, 8, 4};
  int known_lo = 52;   // bits [known_lo, 64) are fixed
  for (int pass = 0; pass < 7; ++pass) {
    const int sh = shifts[pass], wb = widths[pass];
    const uint64_t pre = s_prefix;
    if (s_count == 1) break;
    for (int i = threadIdx.x; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kSelThreads) {
      const uint64_t v = get(i);
      if ((v >> known_lo) == (pre >> known_lo)) atomicAdd(&hist[(v >> sh) & ((1u << wb) - 1)], 1u);
    }
    __syncthreads();
    // 256 bins, one per thread: find the digit holding s_rank
    const uint32_t c = hist[threadIdx.x];
    uint32_t total;
    const uint32_t before = block_exclusive_scan<kSelThreads>(c, scratch, &total);
    const uint32_t r = s_rank;
    __syncthreads();
    if (before < r && r <= before + c) {
      s_prefix = pre | ((uint64_t)threadIdx.x << sh);
      s_rank = r - before;
      s_count = c;
    }
    __syncthreads();
    known_lo = sh;
  }
  if (s_count == 1 && known_lo > 0) {
    // a single item matches the known bits: fetch its full value
    const uint64_t pre = s_prefix;
    for (int i = threadIdx.x; i < n; i += kSelThreads) {
      const uint64_t v = get(i);
      if ((v >> known_lo) == (pre >> known_lo)) s_prefix = v;
    }
    __syncthreads();
  }
  const uint64_t out = s_prefix;
  __syncthreads();
  return out;
}

__global__ void __launch_bounds__(kSelThreads) select_cand_kernel(const SelParams p) {
  __shared__ uint32_t scratch[32];
  __shared__ uint32_t hist[256];
  __shared__ int is_last;
  extern __shared__ uint64_t cand_s[];     // kCandCap composites (last CTA only)
  const int chunk = blockIdx.x, unit = blockIdx.y, b = unit / p.Hkv;
  const UnitInfo ui = unit_info(p, b);
  if (ui.mode == kModeSkip) return;
  const int j0 = chunk * kSelChunk;
  if (j0 >= ui.nb) return;
  uint32_t* st = p.state + (size_t)unit * 8;
  const uint32_t mode = ui.mode;
  const uint32_t bin = __ldcg(&st[kStBin]), count1 = __ldcg(&st[kStCount]);
  const float* sc = p.scores + (size_t)unit * p.n_max;
  uint32_t* cand = p.cand + (size_t)unit * kCandCap * 2;
  uint32_t def = 0;
  for (int i = 0; i < kPerThread; ++i) {
    const int j = j0 + i * kSelThreads + threadIdx.x;
    if (j >= ui.nb) break;
    if (mode == kModeKeepAll) { ++def; continue; }
    const uint32_t key = f2ord(sc[j]), top = key >> 20;
    if (top > bin) {
      ++def;
    } else if (top == bin && count1 <= (uint32_t)kCandCap) {
      const uint32_t slot = atomicAdd(&p.cand_cnt[unit], 1u);
      if (slot < (uint32_t)kCandCap) { cand[slot * 2] = key; cand[slot * 2 + 1] = (uint32_t)j; }
    }
  }
  uint32_t total;
  block_exclusive_scan<kSelThreads>(def, scratch, &total);
  if (threadIdx.x == 0) atomicAdd(&p.chunk_kept[(size_t)unit * p.chunks + chunk], total);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t t = atomicAdd(&p.tickets[unit * 2 + 1], 1u);
    is_last = (t == (uint32_t)ceil_div(ui.nb, kSelChunk) - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  uint64_t thr = 0;   // composite (key << 32 | position) of the k-th smallest slot
  if (mode == kModeNormal) {
    const uint32_t rank = __ldcg(&st[kStRank]);
    const uint64_t prefix = (uint64_t)bin << 52;
    if (count1 <= (uint32_t)kCandCap) {
      const int n = (int)count1;
      for (int i = threadIdx.x; i < n; i += kSelThreads)
        cand_s[i] = ((uint64_t)__ldcg(&cand[i * 2]) << 32) | __ldcg(&cand[i * 2 + 1]);
      __syncthreads();
      thr = radix_select_52(n, rank, prefix, [&](int i) { return cand_s[i]; }, hist, scratch);
      // kept members of the bin, per chunk
      for (int i = threadIdx.x; i < n; i += kSelThreads)
        if (cand_s[i] > thr) atomicAdd(&p.chunk_kept[(size_t)unit * p.chunks + (int)(cand_s[i] & 0xFFFFFFFFu) / kSelChunk], 1u);
    } else {
      // large bin: resolve directly over the head's scores (slow path)
      auto get = [&](int j) -> uint64_t { return ((uint64_t)f2ord(__ldcg(&sc[j])) << 32) | (uint32_t)j; };
      thr = radix_select_52(ui.nb, rank, prefix, get, hist, scratch);
      for (int j = threadIdx.x; j < ui.nb; j += kSelThreads) {
        const uint64_t v = get(j);
        if ((v >> 52) == bin && v > thr) atomicAdd(&p.chunk_kept[(size_t)unit * p.chunks + j / kSelChunk], 1u);
      }
    }
  }
  __threadfence();
  __syncthreads();
  // chunk offsets: exclusive scan of the per-chunk kept counts
  const int nchunks = ceil_div(ui.nb, kSelChunk);
  uint32_t carry = 0;
  for (int c0 = 0; c0 < nchunks; c0 += kSelThreads) {
    const int c = c0 + threadIdx.x;
    const uint32_t v = (c < nchunks) ? __ldcg(&p.chunk_kept[(size_t)unit * p.chunks + c]) : 0u;
    uint32_t tot;
    const uint32_t pre = block_exclusive_scan<kSelThreads>(v, scratch, &tot);
    if (c < nchunks) p.chunk_off[(size_t)unit * p.chunks + c] = carry + pre;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    st[kStKey] = (uint32_t)(thr >> 32);
    st[kStIdx] = (uint32_t)(thr & 0xFFFFFFFFu);
    const uint32_t expect = (uint32_t)(ui.nb - (mode == kModeNormal ? ui.kb : 0));
    if (carry != expect) atomicOr(p.status, DROPKV_FLAG_INTERNAL);
    p.tickets[unit * 2 + 1] = 0;
  }
}

__global__ void __launch_bounds__(kSelThreads) select_write_kernel(const SelParams p) {
  __shared__ uint32_t scratch[32];
  const int chunk = blockIdx.x, unit = blockIdx.y, b = unit / p.Hkv, h = unit - b * p.Hkv;
  const UnitInfo ui = unit_info(p, b);
  if (chunk == 0 && h == 0 && threadIdx.x == 0)
    p.kept_len[b] = (ui.mode == kModeSkip) ? 0 : ui.nb - (ui.mode == kModeNormal ? ui.kb : 0);
  if (ui.mode == kModeSkip) return;
  const int j0 = chunk * kSelChunk;
  if (j0 >= ui.nb) return;
  const uint32_t* st = p.state + (size_t)unit * 8;
  const uint64_t thr = ((uint64_t)__ldcg(&st[kStKey]) << 32) | __ldcg(&st[kStIdx]);
  const float* sc = p.scores + (size_t)unit * p.n_max;
  // each thread owns 16 consecutive slots so the output stays in position order
  const int jt = j0 + threadIdx.x * kPerThread;
  uint32_t keepmask = 0, cnt = 0;
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int j = jt + q;
    bool keep = false;
    if (j < ui.nb) {
      keep = (ui.mode == kModeKeepAll) || ((((uint64_t)f2ord(sc[j]) << 32) | (uint32_t)j) > thr);
    }
    keepmask |= (uint32_t)keep << q;
    cnt += keep;
  }
  uint32_t total;
  const uint32_t before = block_exclusive_scan<kSelThreads>(cnt, scratch, &total);
  int32_t* out = p.kept_idx + (size_t)unit * p.n_max + __ldcg(&p.chunk_off[(size_t)unit * p.chunks + chunk]) + before;
#pragma unroll
  for (int q = 0; q < kPerThread; ++q)
    if ((keepmask >> q) & 1) *out++ = jt + q;
}

// ------------------------------------------------------------ compaction
constexpr int kCompactThreads = 256;
constexpr int kRowsPerWarp = 2;
constexpr int kRowsPerBlock = (kCompactThreads / 32) * kRowsPerWarp;

__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const CompactParams p) {
  const int unit = blockIdx.y, b = unit / p.Hkv, h = unit - b * p.Hkv;
  int kl = p.kept_len[b];
  if (kl > p.out_rows) {
    if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) atomicOr(p.status, DROPKV_FLAG_OVERFLOW);
    kl = p.out_rows;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cpr = p.row_bytes / 16;          // 16-byte chunks per row
  const int32_t* idx = p.kept_idx + (size_t)unit * p.n_max;
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int i = blockIdx.x * kRowsPerBlock + warp * kRowsPerWarp + rr;
    if (i >= kl) break;
    const int src = __ldg(&idx[i]);
    if (src < 0 || src >= p.n_max) {
      if (lane == 0) atomicOr(p.status, DROPKV_FLAG_BAD_LENGTH);
      continue;
    }
    const size_t so = ((size_t)unit * p.n_max + src) * p.row_bytes;
    const size_t dof = ((size_t)unit * p.out_rows + i) * p.row_bytes;
    for (int c = lane; c < 2 * cpr; c += 32) {
      const bool is_v = c >= cpr;
      const int cc = is_v ? c - cpr : c;
      const uint4 val = __ldg(reinterpret_cast<const uint4*>((is_v ? p.v : p.k) + so) + cc);
      *(reinterpret_cast<uint4*>((is_v ? p.v_out : p.k_out) + dof) + cc) = val;
    }
  }
}

}  // namespace

cudaError_t launch_pool_protect(const PoolParams& p, cudaStream_t st) {
  dim3 grid((p.n_max + kPoolTile - 1) / kPoolTile, p.B * p.Hkv);
  pool_protect_kernel<<<grid, kPoolThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_select(const SelParams& p, cudaStream_t st) {
  dim3 grid(p.chunks, p.B * p.Hkv);
  select_hist_kernel<<<grid, kSelThreads, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int dyn = kCandCap * (int)sizeof(uint64_t);
  e = cudaFuncSetAttribute(select_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  select_cand_kernel<<<grid, kSelThreads, dyn, st>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  select_write_kernel<<<grid, kSelThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_compact(const CompactParams& p, cudaStream_t st) {
  if (p.out_rows <= 0) return cudaSuccess;
  dim3 grid((p.out_rows + kRowsPerBlock - 1) / kRowsPerBlock, p.B * p.Hkv);
  compact_kernel<<<grid, kCompactThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace dropkv
