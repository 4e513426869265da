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
//   2. select_cand:  CTAs count the slots above that bin per chunk, gather the
//                    bin's members and histogram their next 12 bits; the last
//                    CTA finds the 24-bit prefix of the k-th pair, ranks the
//                    few members sharing it and turns the per-chunk kept
//                    counts into output offsets.
//   3. select_write: each chunk writes its kept positions in ascending order.
#include <cuda_runtime.h>

#include <algorithm>

#include "dropkv_internal.cuh"
#include "sm103_ptx.cuh"

namespace dropkv {
namespace {

constexpr int kSelThreads = 256;
constexpr int kPoolTile = 2048;
constexpr int kPoolThreads = 256;

enum : uint32_t { kModeNormal = 0, kModeKeepAll = 1, kModeSkip = 2 };
enum { kStMode = 0, kStBin = 1, kStRank = 2, kStCount = 3, kStKey = 4, kStIdx = 5 };

// Order-preserving map of a float to an unsigned key (-0.0 is taken as +0.0,
// so equal scores compare equal and fall to the position tie-break).
__device__ __forceinline__ uint32_t f2ord(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
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
  grid_dep_wait();          // the raw scores come from pass 2
  grid_dep_launch();
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

// Four consecutive scores starting at slot j (j % 4 == 0); slots >= nb read as
// +inf and are masked by the caller.  Vector loads when rows are 16-byte aligned.
__device__ __forceinline__ float4 load4(const float* row, int j, int nb, bool vec) {
  if (vec && j + 3 < nb) return __ldg(reinterpret_cast<const float4*>(row + j));
  float4 v;
  v.x = (j < nb) ? __ldg(row + j) : INFINITY;
  v.y = (j + 1 < nb) ? __ldg(row + j + 1) : INFINITY;
  v.z = (j + 2 < nb) ? __ldg(row + j + 2) : INFINITY;
  v.w = (j + 3 < nb) ? __ldg(row + j + 3) : INFINITY;
  return v;
}

// Shared-memory histogram increments for four consecutive slots: runs of
// equal bins (pooling repeats values over neighbouring slots) are added once.
constexpr uint32_t kNoBin = 0xFFFFFFFFu;
__device__ __forceinline__ void hist_add4(uint32_t* h, uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  uint32_t cur = b0, cnt = 1;
  const uint32_t nxt[3] = {b1, b2, b3};
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    if (nxt[i] == cur) {
      ++cnt;
    } else {
      if (cur != kNoBin) atomicAdd(&h[cur], cnt);
      cur = nxt[i];
      cnt = 1;
    }
  }
  if (cur != kNoBin) atomicAdd(&h[cur], cnt);
}

constexpr int kVec = kSelChunk / (4 * kSelThreads);   // float4 loads per thread per chunk

// The bin of a kHistBins histogram (global memory) that holds the k-th
// (1-based) item, the rank of that item inside the bin and the bin's count.
__device__ void find_bin(const uint32_t* gh, uint32_t k, uint32_t* scratch, uint32_t& bin, uint32_t& rank,
                         uint32_t& count) {
  __shared__ uint32_t s_bin, s_rank, s_count;
  constexpr int per = kHistBins / kSelThreads;
  uint32_t cnt[per];
  uint32_t local = 0;
#pragma unroll
  for (int q = 0; q < per; ++q) {
    cnt[q] = __ldcg(&gh[threadIdx.x * per + q]);
    local += cnt[q];
  }
  uint32_t total;
  const uint32_t before = block_exclusive_scan<kSelThreads>(local, scratch, &total);
  if (before < k && k <= before + local) {
    uint32_t c = before;
    for (int q = 0; q < per; ++q) {
      if (c + cnt[q] >= k) {
        s_bin = threadIdx.x * per + q;
        s_rank = k - c;
        s_count = cnt[q];
        break;
      }
      c += cnt[q];
    }
  }
  __syncthreads();
  bin = s_bin;
  rank = s_rank;
  count = s_count;
  __syncthreads();
}

// Clears the selection counters and histograms (they are accumulated with
// atomics by the kernels that follow).
__global__ void __launch_bounds__(256) select_zero_kernel(uint4* base, size_t n16) {
  grid_dep_wait();
  grid_dep_launch();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    base[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Level 1: histogram of the top 12 bits of the score keys of every KV head;
// the last CTA of a head finds the bin that holds the k_b-th smallest key.
__global__ void __launch_bounds__(kSelThreads) select_hist_kernel(const SelParams p) {
  __shared__ uint32_t sh[kHistBins];
  __shared__ uint32_t scratch[32];
  __shared__ int is_last;
  grid_dep_wait();
  grid_dep_launch();
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
  const float* row = p.scores + (size_t)unit * p.n_max;
  const bool vec = (p.n_max & 3) == 0;
  float4 xv[kVec];   // load phase: all of this thread's slots in flight at once
#pragma unroll
  for (int v = 0; v < kVec; ++v) xv[v] = load4(row, j0 + (v * kSelThreads + threadIdx.x) * 4, ui.nb, vec);
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    const int j = j0 + (v * kSelThreads + threadIdx.x) * 4;
    hist_add4(sh, j < ui.nb ? f2ord(xv[v].x) >> 20 : kNoBin, j + 1 < ui.nb ? f2ord(xv[v].y) >> 20 : kNoBin,
              j + 2 < ui.nb ? f2ord(xv[v].z) >> 20 : kNoBin, j + 3 < ui.nb ? f2ord(xv[v].w) >> 20 : kNoBin);
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
  if (ui.mode == kModeNormal) {
    uint32_t bin, rank, count;
    find_bin(gh, (uint32_t)ui.kb, scratch, bin, rank, count);
    if (threadIdx.x == 0) {
      st[kStBin] = bin;
      st[kStRank] = rank;
      st[kStCount] = count;
    }
  }
  if (threadIdx.x == 0) {
    st[kStMode] = ui.mode;
    p.tickets[unit * 2] = 0;
  }
}

// Radix select of the rank-th (1-based) smallest 64-bit composite among `n`
// items whose bits [known_lo, 64) all equal those of `prefix`; `get(i)`
// returns item i.  Resolves the remaining bits with 8-bit digits.
template <typename Get>
__device__ uint64_t radix_select(int n, uint32_t rank, uint64_t prefix, int known_lo, Get get, uint32_t* hist,
                                 uint32_t* scratch) {
  __shared__ uint64_t s_prefix;
  __shared__ uint32_t s_rank, s_count;
  if (threadIdx.x == 0) { s_prefix = prefix; s_rank = rank; s_count = (uint32_t)n; }
  __syncthreads();
  while (known_lo > 0) {
    const uint64_t pre = s_prefix;
    if (s_count == 1) break;
    const int wb = known_lo < 8 ? known_lo : 8, sh = known_lo - wb;
    for (int i = threadIdx.x; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kSelThreads) {
      const uint64_t v = get(i);
      if ((v >> known_lo) == (pre >> known_lo)) atomicAdd(&hist[(v >> sh) & ((1u << wb) - 1)], 1u);
    }
    __syncthreads();
    const uint32_t c = hist[threadIdx.x];          // 256 bins, one per thread
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

constexpr uint32_t kBruteForce = 1024;   // resolve at most this many survivors by direct ranking

// Level 2: every CTA counts its slots above the bin (kept for sure), gathers
// the bin's members and histograms their next 12 key bits; the last CTA of a
// head locates the 24-bit prefix of the k-th pair, ranks the few members that
// share it directly (radix on larger tie sets), and turns the per-chunk kept
// counts into output offsets.
__global__ void __launch_bounds__(kSelThreads) select_cand_kernel(const SelParams p) {
  __shared__ uint32_t sh2[kHistBins];
  __shared__ uint32_t scratch[32];
  __shared__ uint32_t hist[256];
  __shared__ int is_last;
  __shared__ uint32_t n2_s;
  __shared__ uint64_t thr_s;
  extern __shared__ uint64_t cand_s[];     // kCandCap composites (last CTA only)
  grid_dep_wait();
  grid_dep_launch();
  const int chunk = blockIdx.x, unit = blockIdx.y, b = unit / p.Hkv;
  const UnitInfo ui = unit_info(p, b);
  if (ui.mode == kModeSkip) return;
  const int j0 = chunk * kSelChunk;
  if (j0 >= ui.nb) return;
  uint32_t* st = p.state + (size_t)unit * 8;
  const uint32_t mode = ui.mode;
  const uint32_t bin = __ldcg(&st[kStBin]), count1 = __ldcg(&st[kStCount]);
  const bool gather = mode == kModeNormal && count1 <= (uint32_t)kCandCap;
  const float* row = p.scores + (size_t)unit * p.n_max;
  const bool vec = (p.n_max & 3) == 0;
  uint32_t* cand = p.cand + (size_t)unit * kCandCap * 2;
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) sh2[i] = 0;
  __syncthreads();
  uint32_t def = 0, nmem = 0;
  float4 xv[kVec];   // load phase: all of this thread's slots in flight at once
#pragma unroll
  for (int v = 0; v < kVec; ++v) xv[v] = load4(row, j0 + (v * kSelThreads + threadIdx.x) * 4, ui.nb, vec);
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    const int j = j0 + (v * kSelThreads + threadIdx.x) * 4;
    const float xs[4] = {xv[v].x, xv[v].y, xv[v].z, xv[v].w};
    uint32_t b2[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool valid = j + u < ui.nb;
      const uint32_t key = f2ord(xs[u]), top = key >> 20;
      const bool member = valid && mode == kModeNormal && top == bin;
      def += valid && (mode == kModeKeepAll || top > bin);
      nmem += member;
      b2[u] = member ? (key >> 8) & 0xFFFu : kNoBin;
    }
    hist_add4(sh2, b2[0], b2[1], b2[2], b2[3]);
  }
  uint32_t total;
  block_exclusive_scan<kSelThreads>(def, scratch, &total);
  if (threadIdx.x == 0) atomicAdd(&p.chunk_kept[(size_t)unit * p.chunks + chunk], total);
  if (gather) {
    // members of the bin: one range reservation per CTA, then plain stores
    uint32_t nblk;
    const uint32_t before = block_exclusive_scan<kSelThreads>(nmem, scratch, &nblk);
    __shared__ uint32_t base_s;
    if (threadIdx.x == 0) base_s = nblk ? atomicAdd(&p.cand_cnt[unit], nblk) : 0u;
    __syncthreads();
    uint32_t slot = base_s + before;
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      const int j = j0 + (v * kSelThreads + threadIdx.x) * 4;
      const float xs[4] = {xv[v].x, xv[v].y, xv[v].z, xv[v].w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t key = f2ord(xs[u]);
        if (j + u < ui.nb && (key >> 20) == bin) {
          if (slot < (uint32_t)kCandCap) { cand[slot * 2] = key; cand[slot * 2 + 1] = (uint32_t)(j + u); }
          ++slot;
        }
      }
    }
  }
  if (mode == kModeNormal) {
    uint32_t* gh2 = p.hist2 + (size_t)unit * kHistBins;
    for (int i = threadIdx.x; i < kHistBins; i += kSelThreads)
      if (sh2[i]) atomicAdd(&gh2[i], sh2[i]);
  }
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
    const uint32_t rank1 = __ldcg(&st[kStRank]);
    uint32_t bin2, rank2, count2;
    find_bin(p.hist2 + (size_t)unit * kHistBins, rank1, scratch, bin2, rank2, count2);
    const uint32_t pre24 = (bin << 12) | bin2;
    if (gather) {
      // members sharing the 24-bit prefix of the k-th key
      if (threadIdx.x == 0) n2_s = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < (int)count1; i += kSelThreads) {
        const uint32_t key = __ldcg(&cand[i * 2]);
        if ((key >> 8) == pre24) {
          const uint32_t slot = atomicAdd(&n2_s, 1u);
          cand_s[slot] = ((uint64_t)key << 32) | __ldcg(&cand[i * 2 + 1]);
        }
      }
      __syncthreads();
      const int n2 = (int)n2_s;
      if ((uint32_t)n2 <= kBruteForce) {
        // direct ranking: the member with exactly rank2 - 1 smaller members
        for (int i = threadIdx.x; i < n2; i += kSelThreads) {
          const uint64_t c = cand_s[i];
          uint32_t below = 0;
          for (int q = 0; q < n2; ++q) below += cand_s[q] < c;
          if (below == rank2 - 1) thr_s = c;
        }
        __syncthreads();
        thr = thr_s;
      } else {
        thr = radix_select(n2, rank2, (uint64_t)pre24 << 40, 40, [&](int i) { return cand_s[i]; }, hist, scratch);
      }
      // kept members of the level-1 bin, per chunk (counted in shared memory
      // when the chunk count allows, reusing the level-2 histogram's space)
      const int nchunks_b = ceil_div(ui.nb, kSelChunk);
      const bool local_counts = nchunks_b <= kHistBins;
      if (local_counts) {
        for (int i = threadIdx.x; i < nchunks_b; i += kSelThreads) sh2[i] = 0;
        __syncthreads();
      }
      for (int i = threadIdx.x; i < (int)count1; i += kSelThreads) {
        const uint64_t c = ((uint64_t)__ldcg(&cand[i * 2]) << 32) | __ldcg(&cand[i * 2 + 1]);
        if (c > thr) {
          const int ch = (int)(c & 0xFFFFFFFFu) / kSelChunk;
          if (local_counts) atomicAdd(&sh2[ch], 1u);
          else atomicAdd(&p.chunk_kept[(size_t)unit * p.chunks + ch], 1u);
        }
      }
      if (local_counts) {
        __syncthreads();
        for (int i = threadIdx.x; i < nchunks_b; i += kSelThreads)
          if (sh2[i]) atomicAdd(&p.chunk_kept[(size_t)unit * p.chunks + i], sh2[i]);
      }
    } else {
      // large bin: resolve directly over the head's scores (slow path)
      auto get = [&](int j) -> uint64_t { return ((uint64_t)f2ord(__ldcg(&row[j])) << 32) | (uint32_t)j; };
      thr = radix_select(ui.nb, rank2, (uint64_t)pre24 << 40, 40, get, hist, scratch);
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

// Level 3: each chunk writes its kept positions in ascending order.
__global__ void __launch_bounds__(kSelThreads) select_write_kernel(const SelParams p) {
  __shared__ uint32_t scratch[32];
  grid_dep_wait();
  grid_dep_launch();
  const int chunk = blockIdx.x, unit = blockIdx.y, b = unit / p.Hkv, h = unit - b * p.Hkv;
  const UnitInfo ui = unit_info(p, b);
  if (chunk == 0 && h == 0 && threadIdx.x == 0)
    p.kept_len[b] = (ui.mode == kModeSkip) ? 0 : ui.nb - (ui.mode == kModeNormal ? ui.kb : 0);
  if (ui.mode == kModeSkip) return;
  const int j0 = chunk * kSelChunk;
  if (j0 >= ui.nb) return;
  const uint32_t* st = p.state + (size_t)unit * 8;
  const uint64_t thr = ((uint64_t)__ldcg(&st[kStKey]) << 32) | __ldcg(&st[kStIdx]);
  const float* row = p.scores + (size_t)unit * p.n_max;
  const bool vec = (p.n_max & 3) == 0;
  // each thread owns kPerThread consecutive slots so the output stays in position order
  constexpr int kPer = kSelChunk / kSelThreads;
  const int jt = j0 + threadIdx.x * kPer;
  uint64_t keepmask = 0;
  uint32_t cnt = 0;
  float4 xv[kPer / 4];   // load phase: all of this thread's slots in flight at once
#pragma unroll
  for (int q4 = 0; q4 < kPer / 4; ++q4) xv[q4] = load4(row, jt + q4 * 4, ui.nb, vec);
#pragma unroll
  for (int q4 = 0; q4 < kPer / 4; ++q4) {
    const int j = jt + q4 * 4;
    const float xs[4] = {xv[q4].x, xv[q4].y, xv[q4].z, xv[q4].w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool keep = (j + u < ui.nb) &&
                        ((ui.mode == kModeKeepAll) || ((((uint64_t)f2ord(xs[u]) << 32) | (uint32_t)(j + u)) > thr));
      keepmask |= (uint64_t)keep << (q4 * 4 + u);
      cnt += keep;
    }
  }
  uint32_t total;
  const uint32_t before = block_exclusive_scan<kSelThreads>(cnt, scratch, &total);
  int32_t* out = p.kept_idx + (size_t)unit * p.n_max + __ldcg(&p.chunk_off[(size_t)unit * p.chunks + chunk]) + before;
  while (keepmask) {
    const int q = __ffsll((long long)keepmask) - 1;
    *out++ = jt + q;
    keepmask &= keepmask - 1;
  }
}

// ------------------------------------------------------------ cluster selection
// The whole selection of a KV head inside one thread-block cluster: one CTA
// per 16384-slot chunk (up to 8 chunks), 1024 threads holding 16 consecutive
// slots each in registers.  The k-th pair (T, t) is found digit by digit —
// key bits 31..20, 19..8, 7..0, then the tie rank among slots whose key is T.
// Each digit's histogram is built in shared memory, then its nonzero bins are
// added into every CTA's merged copy with distributed-shared-memory
// reductions (fire and forget), so one cluster barrier per digit completes
// the merged histogram in every CTA and the k-th item's bin is found from
// local shared memory.  No global scratch and a single launch.
constexpr int kClThreads = 1024;
// Slots per thread (PER) of the cluster selection: 4, 8 or 16 consecutive
// slots, a chunk of PER * 1024 slots per CTA.  The launch takes the smallest
// PER whose chunks cover the head with at most kClMax CTAs, so shorter heads
// are spread over more SMs (at n = 32K, 8 CTAs of 4096 slots instead of 2 of
// 16384).
constexpr int kClMax = 8;                        // portable cluster size

struct ClusterSmem {
  uint32_t hist[kHistBins];   // this CTA's histogram of the current digit
  uint32_t mg1[kHistBins];    // merged digit-1 bins (the sums of every CTA's histogram)
  uint32_t mg2[kHistBins];    // merged digit-2 bins
  uint32_t mg3[256];          // merged digit-3 bins
  uint32_t scratch[32];
  uint32_t bc[3];
  uint32_t xch[2 * kClMax];   // (slots above T, slots equal to T) of every CTA of the cluster
};
// Extra shared memory when the selection also pools: the chunk's raw scores
// with a halo of kClHalo >= kMaxPool / 2 slots on each side (a multiple of 4,
// so the chunk itself is 16-byte aligned for vector copies).
constexpr int kClHalo = 32;
static_assert(kClHalo >= kMaxPool / 2 && kClHalo % 4 == 0, "pooling halo");
constexpr size_t kClPoolOff = (sizeof(ClusterSmem) + 15) & ~size_t(15);   // 16-byte aligned for float4 reads
constexpr size_t cl_smem_bytes(int per, bool pool) {
  return pool ? kClPoolOff + (size_t)(per * kClThreads + 2 * kClHalo) * sizeof(float) : sizeof(ClusterSmem);
}

// Cluster barrier halves (every thread of every CTA of the cluster arrives;
// release / acquire order the shared-memory accesses around it).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_barrier() {
  cluster_arrive();
  cluster_wait();
}

// Address of `local` (this CTA's shared memory) in the shared memory of the
// cluster's CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(local)), "r"(rank));
  return out;
}
__device__ __forceinline__ void cluster_red_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_store(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Adds the nonzero bins of the local histogram into every CTA's merged copy.
template <int BINS>
__device__ __forceinline__ void cluster_push(const uint32_t* hist, uint32_t* merged, int C) {
  for (int i = threadIdx.x; i < BINS; i += kClThreads) {
    const uint32_t c = hist[i];
    if (c)
      for (int dst = 0; dst < C; ++dst) cluster_red_add(cluster_map(merged + i, (uint32_t)dst), c);
  }
}

// Bin of the merged shared-memory histogram that holds the k-th (1-based)
// item, the item's rank inside the bin and the bin's count.
template <int BINS>
__device__ __forceinline__ void cluster_find_bin(const uint32_t* merged, uint32_t k, uint32_t* scratch, uint32_t* bc,
                                                 uint32_t& bin, uint32_t& rank, uint32_t& count) {
  constexpr int per = BINS >= kClThreads ? BINS / kClThreads : 1;
  const int base = (int)threadIdx.x * per;
  uint32_t cnt[per];
  uint32_t local = 0;
#pragma unroll
  for (int q = 0; q < per; ++q) {
    cnt[q] = (base + q < BINS) ? merged[base + q] : 0u;
    local += cnt[q];
  }
  if (threadIdx.x == 0) { bc[0] = 0; bc[1] = 1; bc[2] = 0; }
  uint32_t total;
  const uint32_t before = block_exclusive_scan<kClThreads>(local, scratch, &total);
  if (before < k && k <= before + local) {
    uint32_t c = before;
#pragma unroll
    for (int q = 0; q < per; ++q) {
      if (c < k && k <= c + cnt[q]) { bc[0] = base + q; bc[1] = k - c; bc[2] = cnt[q]; }
      c += cnt[q];
    }
  }
  __syncthreads();
  bin = bc[0];
  rank = bc[1];
  count = bc[2];
  __syncthreads();
}

// Run-aggregated shared-memory histogram of this thread's slots: slot u adds
// to bin `digit(key)` when u < nv and `member(key)`.
template <int PER, typename Member, typename Digit>
__device__ __forceinline__ void cluster_hist_add(uint32_t* hist, const uint32_t (&key)[PER], int nv, Member member,
                                                 Digit digit) {
  uint32_t cur = kNoBin, cnt = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const uint32_t bn = (u < nv && member(key[u])) ? digit(key[u]) : kNoBin;
    if (bn == cur) {
      ++cnt;
    } else {
      if (cur != kNoBin) atomicAdd(&hist[cur], cnt);
      cur = bn;
      cnt = 1;
    }
  }
  if (cur != kNoBin) atomicAdd(&hist[cur], cnt);
}

template <int PER>
__global__ void __launch_bounds__(kClThreads, 1) select_cluster_kernel(const SelParams p) {
  constexpr int kClPer = PER, kChunk = PER * kClThreads;
  extern __shared__ __align__(16) uint8_t cl_smem_raw[];
  ClusterSmem& S = *reinterpret_cast<ClusterSmem*>(cl_smem_raw);
  // the cluster spans blockIdx.x (its dimension is gridDim.x), so the rank
  // of a CTA in its cluster is its chunk index
  const int C = (int)gridDim.x, r = (int)blockIdx.x, unit = blockIdx.y, b = unit / p.Hkv, h = unit - b * p.Hkv;
  // lengths and k are caller inputs that no kernel of the path writes: read
  // them, and clear the merge bins, while the scores are still being made
  const UnitInfo ui = unit_info(p, b);
  const bool normal = ui.mode == kModeNormal;
  if (normal) {
    for (int i = threadIdx.x; i < kHistBins; i += kClThreads) S.hist[i] = S.mg1[i] = S.mg2[i] = 0u;
    if (threadIdx.x < 256) S.mg3[threadIdx.x] = 0u;
    // first barrier, split: arrive now (bins cleared), wait before the first
    // access to another CTA, so its latency hides behind the loads
    cluster_arrive();
  }
  grid_dep_wait();
  grid_dep_launch();
  if (r == 0 && h == 0 && threadIdx.x == 0) {
    if (ui.mode == kModeSkip) atomicOr(p.status, DROPKV_FLAG_BAD_LENGTH);
    else if (ui.kb < 0 || ui.kb > ui.nb - p.protect) atomicOr(p.status, DROPKV_FLAG_BAD_K);
    p.kept_len[b] = (ui.mode == kModeSkip) ? 0 : ui.nb - (normal ? ui.kb : 0);
  }
  const int nb = (ui.mode == kModeSkip) ? 0 : ui.nb;
  const int jt = r * kChunk + (int)threadIdx.x * kClPer;
  const int nv = min(max(nb - jt, 0), kClPer);
  int32_t* out_row = p.kept_idx + (size_t)unit * p.n_max;
  const bool vec = (p.n_max & 3) == 0;
  uint32_t key[kClPer];
  bool have_keys = false;
  if (p.pool.raw) {
    // MaxPool1D (window clipped to [0, n_b)) then protection of the last
    // `protect` slots, as pool_protect_kernel; skipped for lengths that
    // kernel rejects (the window statistics flag them)
    const int pnb = ui.nb;   // lengths[b] (or n_max), read before the wait
    if (pnb >= p.pool.w && pnb <= p.n_max) {
      // buf[i] = raw[j0 - kClHalo + i]; -inf outside [0, n_b)
      float* buf = reinterpret_cast<float*>(cl_smem_raw + kClPoolOff);
      const int half = p.pool.half, j0 = r * kChunk;
      const float* raw = p.pool.raw + (size_t)unit * p.n_max;
      float4 x[kClPer / 4];
#pragma unroll
      for (int q = 0; q < kClPer / 4; ++q) {
        const int j = j0 + 4 * ((int)threadIdx.x + q * kClThreads);
        if (vec && j + 3 < pnb) {
          x[q] = __ldg(reinterpret_cast<const float4*>(raw + j));
        } else {
          x[q].x = (j < pnb) ? __ldg(raw + j) : -INFINITY;
          x[q].y = (j + 1 < pnb) ? __ldg(raw + j + 1) : -INFINITY;
          x[q].z = (j + 2 < pnb) ? __ldg(raw + j + 2) : -INFINITY;
          x[q].w = (j + 3 < pnb) ? __ldg(raw + j + 3) : -INFINITY;
        }
      }
      if (threadIdx.x < 2 * kClHalo) {
        const int i = threadIdx.x < kClHalo ? (int)threadIdx.x : kChunk + (int)threadIdx.x;
        const int jj = j0 - kClHalo + i;
        buf[i] = (jj >= 0 && jj < pnb) ? __ldg(raw + jj) : -INFINITY;
      }
#pragma unroll
      for (int q = 0; q < kClPer / 4; ++q)
        *reinterpret_cast<float4*>(buf + kClHalo + 4 * ((int)threadIdx.x + q * kClThreads)) = x[q];
      __syncthreads();
      // this thread's 16 consecutive slots, from the 16 + 2 * half values around them
      const int base = kClHalo + (int)threadIdx.x * kClPer;
      float pv[kClPer];
      if (half <= 4) {
        float wv[kClPer + 8];
#pragma unroll
        for (int c = 0; c < (kClPer + 8) / 4; ++c) {
          const float4 t = *reinterpret_cast<const float4*>(buf + base - 4 + 4 * c);
          wv[4 * c] = t.x; wv[4 * c + 1] = t.y; wv[4 * c + 2] = t.z; wv[4 * c + 3] = t.w;
        }
#pragma unroll
        for (int u = 0; u < kClPer; ++u) {
          float m = wv[4 + u];
#pragma unroll
          for (int t = 1; t <= 4; ++t)
            if (t <= half) m = fmaxf(m, fmaxf(wv[4 + u - t], wv[4 + u + t]));
          pv[u] = m;
        }
      } else {
#pragma unroll
        for (int u = 0; u < kClPer; ++u) {
          float m = buf[base + u - half];
          for (int t = 1; t <= 2 * half; ++t) m = fmaxf(m, buf[base + u - half + t]);
          pv[u] = m;
        }
      }
      const int first_protected = pnb - p.protect;
      float* out = p.pool.scores + (size_t)unit * p.n_max + jt;
#pragma unroll
      for (int u = 0; u < kClPer; ++u) pv[u] = (jt + u >= first_protected) ? INFINITY : pv[u];
      if (vec && jt + kClPer <= pnb) {
#pragma unroll
        for (int q = 0; q < kClPer / 4; ++q)
          reinterpret_cast<float4*>(out)[q] = make_float4(pv[4 * q], pv[4 * q + 1], pv[4 * q + 2], pv[4 * q + 3]);
      } else {
#pragma unroll
        for (int u = 0; u < kClPer; ++u)
          if (jt + u < pnb) out[u] = pv[u];
      }
#pragma unroll
      for (int u = 0; u < kClPer; ++u) key[u] = f2ord(pv[u]);
      have_keys = true;
    }
  }
  if (!normal) {
    // nothing evicted: kept slot j sits at index j (the branch is uniform over the cluster)
    for (int u = 0; u < nv; ++u) out_row[jt + u] = jt + u;
    return;
  }
  if (!have_keys) {
    const float* row = p.scores + (size_t)unit * p.n_max;
#pragma unroll
    for (int q4 = 0; q4 < kClPer / 4; ++q4) {
      const float4 x = load4(row, jt + q4 * 4, nb, vec);
      key[q4 * 4 + 0] = f2ord(x.x);
      key[q4 * 4 + 1] = f2ord(x.y);
      key[q4 * 4 + 2] = f2ord(x.z);
      key[q4 * 4 + 3] = f2ord(x.w);
    }
  }
  __syncthreads();   // cleared bins

  // digit 1: key bits 31..20
  cluster_hist_add(S.hist, key, nv, [](uint32_t) { return true; }, [](uint32_t k) { return k >> 20; });
  __syncthreads();
  cluster_wait();    // every CTA of the cluster running, its merged bins cleared
  cluster_push<kHistBins>(S.hist, S.mg1, C);
  cluster_barrier();
  uint32_t bin1, rank1, cnt1;
  cluster_find_bin<kHistBins>(S.mg1, (uint32_t)ui.kb, S.scratch, S.bc, bin1, rank1, cnt1);

  // digit 2: key bits 19..8 of the members of bin1
  for (int i = threadIdx.x; i < kHistBins; i += kClThreads) S.hist[i] = 0;
  __syncthreads();
  cluster_hist_add(S.hist, key, nv, [bin1](uint32_t k) { return (k >> 20) == bin1; },
                   [](uint32_t k) { return (k >> 8) & 0xFFFu; });
  __syncthreads();
  cluster_push<kHistBins>(S.hist, S.mg2, C);
  cluster_barrier();
  uint32_t bin2, rank2, cnt2;
  cluster_find_bin<kHistBins>(S.mg2, rank1, S.scratch, S.bc, bin2, rank2, cnt2);
  const uint32_t pre24 = (bin1 << 12) | bin2;

  // digit 3: key bits 7..0 of the members sharing the 24-bit prefix
  for (int i = threadIdx.x; i < 256; i += kClThreads) S.hist[i] = 0;
  __syncthreads();
  cluster_hist_add(S.hist, key, nv, [pre24](uint32_t k) { return (k >> 8) == pre24; },
                   [](uint32_t k) { return k & 0xFFu; });
  __syncthreads();
  cluster_push<256>(S.hist, S.mg3, C);
  cluster_barrier();
  uint32_t bin3, rank3, cnt3;
  cluster_find_bin<256>(S.mg3, rank2, S.scratch, S.bc, bin3, rank3, cnt3);
  const uint32_t T = (pre24 << 8) | bin3;

  // tie rank: the slots with key T are evicted in position order up to rank3
  uint32_t above = 0, ties = 0;
#pragma unroll
  for (int u = 0; u < kClPer; ++u) {
    above += (u < nv && key[u] > T);
    ties += (u < nv && key[u] == T);
  }
  uint32_t packed_total;   // (above << 16 | ties); a chunk holds at most 16384 slots
  const uint32_t packed_before = block_exclusive_scan<kClThreads>((above << 16) | ties, S.scratch, &packed_total);
  if (threadIdx.x < (unsigned)C) {
    cluster_store(cluster_map(S.xch + 2 * r, threadIdx.x), packed_total >> 16);
    cluster_store(cluster_map(S.xch + 2 * r + 1, threadIdx.x), packed_total & 0xFFFFu);
  }
  cluster_barrier();   // last access to another CTA's shared memory is before this point
  // offsets of this CTA among the ties and among the kept slots of the head
  uint32_t tie_pre = 0, kept_pre = 0, tie_off = 0, kept_off = 0;
  for (int s = 0; s < C; ++s) {
    const uint32_t a = S.xch[2 * s], t = S.xch[2 * s + 1];
    const int past = (int)(tie_pre + t) - (int)rank3;   // ties of CTA s ranked after rank3
    if (s == r) { tie_off = tie_pre; kept_off = kept_pre; }
    tie_pre += t;
    kept_pre += a + (uint32_t)min(max(past, 0), (int)t);
  }
  if (r == 0 && threadIdx.x == 0 && kept_pre != (uint32_t)(nb - ui.kb)) atomicOr(p.status, DROPKV_FLAG_INTERNAL);
  // kept slots of the earlier threads of this CTA: all their slots above T,
  // and their ties ranked after rank3 (tie ranks tie_off + 1 .. tie_off + tb)
  const uint32_t ab = packed_before >> 16, tb = packed_before & 0xFFFFu;
  const int tb_kept = min(max((int)(tie_off + tb) - (int)rank3, 0), (int)tb);
  uint32_t tr = tie_off + tb;   // tie rank before this thread's slots
  uint32_t keepmask = 0;
#pragma unroll
  for (int u = 0; u < kClPer; ++u) {
    const bool eq = u < nv && key[u] == T;
    tr += eq;
    const bool keep = u < nv && (key[u] > T || (eq && tr > rank3));
    keepmask |= (uint32_t)keep << u;
  }
  int32_t* out = out_row + kept_off + ab + (uint32_t)tb_kept;
  while (keepmask) {
    const int q = __ffs((int)keepmask) - 1;
    *out++ = jt + q;
    keepmask &= keepmask - 1;
  }
}

// ------------------------------------------------------------ layer-wide selection
// The adaptive head budget of AdaDropKV ("DropKV: Decoupling ...", section 5.3
// and Appendix A.3), read as one pool per sequence: the scores of all its KV
// heads compete, and the evict_total[b] smallest (score, head, position)
// triples are evicted, so each head keeps its own number of slots.  Grid
// (chunks, Hkv, B): one 4096-slot chunk of one head per CTA (many CTAs: each
// kernel is short and latency-bound), 16 consecutive slots per thread.  The k-th triple is found digit by digit (key bits
// 31..20, 19..8, 7..0, then the tie rank among equal keys in head-major
// order) over five kernels whose boundaries order the global histograms, so
// nothing waits on another CTA; the last kernel turns per-chunk counts into
// per-head output offsets.
enum { kLsBin1 = 0, kLsRank1 = 1, kLsPre24 = 2, kLsRank2 = 3, kLsKey = 4, kLsRank3 = 5 };
constexpr int kLsPer = kLayerChunk / kSelThreads;   // 16 consecutive slots per thread

struct LayerInfo {
  int nb, e;
  uint32_t mode;
};

__device__ __forceinline__ LayerInfo layer_info(const LayerSelParams& p, int b) {
  LayerInfo u;
  u.nb = p.lengths ? p.lengths[b] : p.n_max;
  u.e = p.evict_total[b];
  if (u.nb < 1 || u.nb > p.n_max || u.nb < p.protect) u.mode = kModeSkip;
  else if (u.e <= 0 || (long long)u.e > (long long)p.Hkv * (u.nb - p.protect)) u.mode = kModeKeepAll;
  else u.mode = kModeNormal;
  return u;
}

// Keys of this thread's slots j0 + 16 t + [0, 16) (slots >= nb are masked by nv).
__device__ __forceinline__ int layer_keys(const LayerSelParams& p, int b, int h, int j0, int nb,
                                          uint32_t (&key)[kLsPer]) {
  const float* row = p.scores + ((size_t)b * p.Hkv + h) * p.n_max;
  const bool vec = (p.n_max & 3) == 0;
  const int jt = j0 + (int)threadIdx.x * kLsPer;
#pragma unroll
  for (int q4 = 0; q4 < kLsPer / 4; ++q4) {
    const float4 x = load4(row, jt + q4 * 4, nb, vec);
    key[q4 * 4 + 0] = f2ord(x.x);
    key[q4 * 4 + 1] = f2ord(x.y);
    key[q4 * 4 + 2] = f2ord(x.z);
    key[q4 * 4 + 3] = f2ord(x.w);
  }
  return min(max(nb - jt, 0), kLsPer);
}

// Run-aggregated shared-memory histogram of the slots u < nv with member(key).
template <typename Member, typename Digit>
__device__ __forceinline__ void layer_hist_add(uint32_t* hist, const uint32_t (&key)[kLsPer], int nv, Member member,
                                               Digit digit) {
  uint32_t cur = kNoBin, cnt = 0;
#pragma unroll
  for (int u = 0; u < kLsPer; ++u) {
    const uint32_t bn = (u < nv && member(key[u])) ? digit(key[u]) : kNoBin;
    if (bn == cur) {
      ++cnt;
    } else {
      if (cur != kNoBin) atomicAdd(&hist[cur], cnt);
      cur = bn;
      cnt = 1;
    }
  }
  if (cur != kNoBin) atomicAdd(&hist[cur], cnt);
}

template <int BINS>
__device__ __forceinline__ void layer_flush(const uint32_t* sh, uint32_t* gh) {
  __syncthreads();
  for (int i = threadIdx.x; i < BINS; i += kSelThreads)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
}

// Digit 1 (key bits 31..20) of every head of the sequence into one histogram.
__global__ void __launch_bounds__(kSelThreads) layer_hist1_kernel(const LayerSelParams p) {
  __shared__ uint32_t sh[kHistBins];
  grid_dep_wait();
  grid_dep_launch();
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const LayerInfo li = layer_info(p, b);
  if (chunk == 0 && h == 0 && threadIdx.x == 0) {
    if (li.mode == kModeSkip) atomicOr(p.status, DROPKV_FLAG_BAD_LENGTH);
    else if (li.e < 0 || (long long)li.e > (long long)p.Hkv * (li.nb - p.protect)) atomicOr(p.status, DROPKV_FLAG_BAD_K);
  }
  const int j0 = chunk * kLayerChunk;
  if (li.mode != kModeNormal || j0 >= li.nb) return;
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) sh[i] = 0;
  __syncthreads();
  uint32_t key[kLsPer];
  const int nv = layer_keys(p, b, h, j0, li.nb, key);
  layer_hist_add(sh, key, nv, [](uint32_t) { return true; }, [](uint32_t k) { return k >> 20; });
  layer_flush<kHistBins>(sh, p.h1 + (size_t)b * kHistBins);
}

// Digit 2 (key bits 19..8) of the members of the k-th key's digit-1 bin.
__global__ void __launch_bounds__(kSelThreads) layer_hist2_kernel(const LayerSelParams p) {
  __shared__ uint32_t sh[kHistBins];
  __shared__ uint32_t scratch[32];
  grid_dep_wait();
  grid_dep_launch();
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const LayerInfo li = layer_info(p, b);
  const int j0 = chunk * kLayerChunk;
  if (li.mode != kModeNormal || j0 >= li.nb) return;
  uint32_t bin1, rank1, cnt1;
  find_bin(p.h1 + (size_t)b * kHistBins, (uint32_t)li.e, scratch, bin1, rank1, cnt1);
  if (chunk == 0 && h == 0 && threadIdx.x == 0) {
    p.state[b * 8 + kLsBin1] = bin1;
    p.state[b * 8 + kLsRank1] = rank1;
  }
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) sh[i] = 0;
  __syncthreads();
  uint32_t key[kLsPer];
  const int nv = layer_keys(p, b, h, j0, li.nb, key);
  layer_hist_add(sh, key, nv, [bin1](uint32_t k) { return (k >> 20) == bin1; },
                 [](uint32_t k) { return (k >> 8) & 0xFFFu; });
  layer_flush<kHistBins>(sh, p.h2 + (size_t)b * kHistBins);
}

// Digit 3 (key bits 7..0) of the members sharing the k-th key's 24-bit prefix.
__global__ void __launch_bounds__(kSelThreads) layer_hist3_kernel(const LayerSelParams p) {
  __shared__ uint32_t sh[256];
  __shared__ uint32_t scratch[32];
  grid_dep_wait();
  grid_dep_launch();
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const LayerInfo li = layer_info(p, b);
  const int j0 = chunk * kLayerChunk;
  if (li.mode != kModeNormal || j0 >= li.nb) return;
  const uint32_t bin1 = __ldcg(&p.state[b * 8 + kLsBin1]), rank1 = __ldcg(&p.state[b * 8 + kLsRank1]);
  uint32_t bin2, rank2, cnt2;
  find_bin(p.h2 + (size_t)b * kHistBins, rank1, scratch, bin2, rank2, cnt2);
  const uint32_t pre24 = (bin1 << 12) | bin2;
  if (chunk == 0 && h == 0 && threadIdx.x == 0) {
    p.state[b * 8 + kLsPre24] = pre24;
    p.state[b * 8 + kLsRank2] = rank2;
  }
  sh[threadIdx.x] = 0;   // 256 threads, 256 bins
  __syncthreads();
  uint32_t key[kLsPer];
  const int nv = layer_keys(p, b, h, j0, li.nb, key);
  layer_hist_add(sh, key, nv, [pre24](uint32_t k) { return (k >> 8) == pre24; }, [](uint32_t k) { return k & 0xFFu; });
  layer_flush<256>(sh, p.h3 + (size_t)b * 256);
}

// The k-th key T and its rank among the equal keys; per chunk, the slots
// above T and equal to T (written for every chunk, zero past the sequence).
__global__ void __launch_bounds__(kSelThreads) layer_count_kernel(const LayerSelParams p) {
  static_assert(kSelThreads == 256, "one digit-3 bin per thread");
  __shared__ uint32_t scratch[32];
  __shared__ uint32_t t_s, r_s;
  grid_dep_wait();
  grid_dep_launch();
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const LayerInfo li = layer_info(p, b);
  if (li.mode != kModeNormal) return;
  const int j0 = chunk * kLayerChunk;
  uint32_t* cnt_out = p.counts + (((size_t)b * p.Hkv + h) * p.chunks + chunk) * 2;
  if (j0 >= li.nb) {
    if (threadIdx.x == 0) { cnt_out[0] = 0; cnt_out[1] = 0; }
    return;
  }
  const uint32_t pre24 = __ldcg(&p.state[b * 8 + kLsPre24]), rank2 = __ldcg(&p.state[b * 8 + kLsRank2]);
  const uint32_t c3 = __ldcg(&p.h3[(size_t)b * 256 + threadIdx.x]);
  if (threadIdx.x == 0) { t_s = pre24 << 8; r_s = 1; }
  uint32_t total;
  const uint32_t before = block_exclusive_scan<kSelThreads>(c3, scratch, &total);
  if (before < rank2 && rank2 <= before + c3) {
    t_s = (pre24 << 8) | threadIdx.x;
    r_s = rank2 - before;
  }
  __syncthreads();
  const uint32_t T = t_s, rank3 = r_s;
  if (chunk == 0 && h == 0 && threadIdx.x == 0) {
    p.state[b * 8 + kLsKey] = T;
    p.state[b * 8 + kLsRank3] = rank3;
  }
  uint32_t key[kLsPer];
  const int nv = layer_keys(p, b, h, j0, li.nb, key);
  uint32_t above = 0, ties = 0;
#pragma unroll
  for (int u = 0; u < kLsPer; ++u) {
    above += (u < nv && key[u] > T);
    ties += (u < nv && key[u] == T);
  }
  uint32_t packed_total;   // (above << 16) | ties; a chunk holds at most 4096 slots
  block_exclusive_scan<kSelThreads>((above << 16) | ties, scratch, &packed_total);
  if (threadIdx.x == 0) {
    cnt_out[0] = packed_total >> 16;
    cnt_out[1] = packed_total & 0xFFFFu;
  }
}

// Kept positions of every head, ascending, and the per-head kept counts.
__global__ void __launch_bounds__(kSelThreads) layer_write_kernel(const LayerSelParams p) {
  __shared__ uint32_t scratch[32];
  __shared__ uint32_t tie_off_s, head_off_s, kfirst_s, klast_s;
  grid_dep_wait();
  grid_dep_launch();
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const LayerInfo li = layer_info(p, b);
  const int j0 = chunk * kLayerChunk;
  int32_t* out_row = p.kept_idx + ((size_t)b * p.Hkv + h) * p.n_max;
  int32_t* kept_len = p.kept_len + (size_t)b * p.Hkv + h;
  if (li.mode == kModeSkip) {
    if (chunk == 0 && threadIdx.x == 0) *kept_len = 0;
    return;
  }
  if (li.mode == kModeKeepAll) {
    if (chunk == 0 && threadIdx.x == 0) *kept_len = li.nb;
    for (int j = j0 + threadIdx.x; j < min(j0 + kLayerChunk, li.nb); j += kSelThreads) out_row[j] = j;
    return;
  }
  const uint32_t T = __ldcg(&p.state[b * 8 + kLsKey]), rank3 = __ldcg(&p.state[b * 8 + kLsRank3]);
  {
    // per-chunk (above, tie) counts in head-major order, scanned 256 at a time:
    // the tie offset of this chunk, the kept slots of this head before it, and
    // (chunk 0) the head's kept count
    const uint32_t* cnt = p.counts + (size_t)b * p.Hkv * p.chunks * 2;
    const int n = p.Hkv * p.chunks, mine = h * p.chunks + chunk;
    const int head_first = h * p.chunks, head_last = head_first + p.chunks - 1;
    uint32_t carry_t = 0, carry_k = 0;
    for (int base = 0; base < n; base += kSelThreads) {
      const int e = base + (int)threadIdx.x;
      const uint32_t a = e < n ? __ldcg(&cnt[(size_t)e * 2]) : 0u;
      const uint32_t t = e < n ? __ldcg(&cnt[(size_t)e * 2 + 1]) : 0u;
      uint32_t tsum, ksum;
      const uint32_t tie_pre = carry_t + block_exclusive_scan<kSelThreads>(t, scratch, &tsum);
      const int past = (int)(tie_pre + t) - (int)rank3;   // ties of this chunk ranked after rank3
      const uint32_t kept_e = a + (uint32_t)min(max(past, 0), (int)t);
      const uint32_t kpre = carry_k + block_exclusive_scan<kSelThreads>(kept_e, scratch, &ksum);
      if (e == mine) { tie_off_s = tie_pre; head_off_s = kpre; }
      if (e == head_first) kfirst_s = kpre;
      if (e == head_last) klast_s = kpre + kept_e;
      carry_t += tsum;
      carry_k += ksum;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      head_off_s -= kfirst_s;
      if (chunk == 0) *kept_len = (int32_t)(klast_s - kfirst_s);
      if (h == 0 && chunk == 0 && (long long)carry_k != (long long)p.Hkv * li.nb - li.e)
        atomicOr(p.status, DROPKV_FLAG_INTERNAL);
    }
  }
  __syncthreads();
  if (j0 >= li.nb) return;
  uint32_t key[kLsPer];
  const int nv = layer_keys(p, b, h, j0, li.nb, key);
  const int jt = j0 + (int)threadIdx.x * kLsPer;
  uint32_t above = 0, ties = 0;
#pragma unroll
  for (int u = 0; u < kLsPer; ++u) {
    above += (u < nv && key[u] > T);
    ties += (u < nv && key[u] == T);
  }
  uint32_t packed_total;
  const uint32_t packed_before = block_exclusive_scan<kSelThreads>((above << 16) | ties, scratch, &packed_total);
  const uint32_t ab = packed_before >> 16, tb = packed_before & 0xFFFFu;
  const uint32_t tie_off = tie_off_s;
  const int tb_kept = min(max((int)(tie_off + tb) - (int)rank3, 0), (int)tb);
  int32_t* out = out_row + head_off_s + ab + (uint32_t)tb_kept;
  uint32_t tr = tie_off + tb;   // tie rank before this thread's slots
#pragma unroll
  for (int u = 0; u < kLsPer; ++u) {
    const bool eq = u < nv && key[u] == T;
    tr += eq;
    if (u < nv && (key[u] > T || (eq && tr > rank3))) *out++ = jt + u;
  }
}

// ------------------------------------------------------------ compaction
constexpr int kCompactThreads = 256;
constexpr int kRowsPerWarp = 2;
constexpr int kRowsPerBlock = (kCompactThreads / 32) * kRowsPerWarp;

__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const CompactParams p) {
  grid_dep_wait();          // kept_idx / kept_len come from the selection
  grid_dep_launch();
  const int unit = blockIdx.y, b = unit / p.Hkv, h = unit - b * p.Hkv;
  int kl = p.per_head ? p.kept_len[unit] : p.kept_len[b];
  if (kl > p.out_rows) {
    if (blockIdx.x == 0 && (h == 0 || p.per_head) && threadIdx.x == 0) atomicOr(p.status, DROPKV_FLAG_OVERFLOW);
    kl = p.out_rows;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cpr = p.row_bytes / 16;          // 16-byte chunks per row
  const int32_t* idx = p.kept_idx + (size_t)unit * p.n_max;
  // grid-stride over the head's kept rows: the grid is sized for the GPU,
  // not for out_rows (which may be far above the kept count).  A row is at
  // most 2 x 16 chunks of 16 bytes (K and V, d <= 128): lane c moves chunk c
  // of both of the warp's rows, loads first.
  static_assert(kRowsPerWarp == 2, "two rows per warp and iteration");
  const bool is_v = lane >= cpr;
  const int cc = is_v ? lane - cpr : lane;
  const uint8_t* src_base = is_v ? p.v : p.k;
  uint8_t* dst_base = is_v ? p.v_out : p.k_out;
  for (int i0 = blockIdx.x * kRowsPerBlock + warp * kRowsPerWarp; i0 < kl; i0 += gridDim.x * kRowsPerBlock) {
    const int i1 = i0 + 1;
    int s0 = __ldg(&idx[i0]);
    int s1 = i1 < kl ? __ldg(&idx[i1]) : 0;
    // an index outside the cache is flagged and its row skipped (clamped so the load stays in bounds)
    const bool bad0 = s0 < 0 || s0 >= p.n_max, bad1 = s1 < 0 || s1 >= p.n_max;
    if ((bad0 || bad1) && lane == 0) atomicOr(p.status, DROPKV_FLAG_BAD_LENGTH);
    s0 = min(max(s0, 0), p.n_max - 1);
    s1 = min(max(s1, 0), p.n_max - 1);
    if (lane < 2 * cpr) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(src_base + ((size_t)unit * p.n_max + s0) * p.row_bytes) + cc);
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(src_base + ((size_t)unit * p.n_max + s1) * p.row_bytes) + cc);
      if (!bad0) *(reinterpret_cast<uint4*>(dst_base + ((size_t)unit * p.out_rows + i0) * p.row_bytes) + cc) = a;
      if (!bad1 && i1 < kl)
        *(reinterpret_cast<uint4*>(dst_base + ((size_t)unit * p.out_rows + i1) * p.row_bytes) + cc) = c;
    }
  }
}

}  // namespace

cudaError_t launch_pool_protect(const PoolParams& p, cudaStream_t st) {
  dim3 grid((p.n_max + kPoolTile - 1) / kPoolTile, p.B * p.Hkv);
  return launch_pdl(pool_protect_kernel, grid, dim3(kPoolThreads), 0, st, p);
}

cudaError_t launch_select(const SelParams& p, size_t zero_bytes, void* zero_base, cudaStream_t st) {
  dim3 grid(p.chunks, p.B * p.Hkv);
  if (p.chunks <= kClMax) {
    // one cluster per KV head: no global counters to clear
    const int per = p.n_max <= kClMax * 4 * kClThreads ? 4 : (p.n_max <= kClMax * 8 * kClThreads ? 8 : 16);
    const int C = (p.n_max + per * kClThreads - 1) / (per * kClThreads);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, p.B * p.Hkv);
    cfg.blockDim = dim3(kClThreads);
    cfg.stream = st;
    cfg.dynamicSmemBytes = cl_smem_bytes(per, p.pool.raw != nullptr);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    auto kern = per == 4 ? select_cluster_kernel<4> : (per == 8 ? select_cluster_kernel<8> : select_cluster_kernel<16>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cl_smem_bytes(per, true));
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e == cudaSuccess) return e;
    (void)cudaGetLastError();   // clusters refused on this device: take the multi-kernel path
  }
  if (p.pool.raw) {
    const cudaError_t e = launch_pool_protect(p.pool, st);
    if (e != cudaSuccess) return e;
  }
  const size_t n16 = zero_bytes / 16;
  const int zb = (int)std::min<size_t>((n16 + 255) / 256, 1024);
  cudaError_t e = launch_pdl(select_zero_kernel, dim3(zb > 0 ? zb : 1), dim3(256), 0, st,
                             reinterpret_cast<uint4*>(zero_base), n16);
  if (e != cudaSuccess) return e;
  e = launch_pdl(select_hist_kernel, grid, dim3(kSelThreads), 0, st, p);
  if (e != cudaSuccess) return e;
  const int dyn = kCandCap * (int)sizeof(uint64_t);
  e = cudaFuncSetAttribute(select_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  e = launch_pdl(select_cand_kernel, grid, dim3(kSelThreads), (size_t)dyn, st, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(select_write_kernel, grid, dim3(kSelThreads), 0, st, p);
}

cudaError_t launch_select_layer(const LayerSelParams& p, size_t zero_bytes, void* zero_base, cudaStream_t st) {
  const size_t n16 = zero_bytes / 16;
  const int zb = (int)std::min<size_t>((n16 + 255) / 256, 1024);
  cudaError_t e = launch_pdl(select_zero_kernel, dim3(zb > 0 ? zb : 1), dim3(256), 0, st,
                             reinterpret_cast<uint4*>(zero_base), n16);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.chunks, p.Hkv, p.B);
  if ((e = launch_pdl(layer_hist1_kernel, grid, dim3(kSelThreads), 0, st, p)) != cudaSuccess) return e;
  if ((e = launch_pdl(layer_hist2_kernel, grid, dim3(kSelThreads), 0, st, p)) != cudaSuccess) return e;
  if ((e = launch_pdl(layer_hist3_kernel, grid, dim3(kSelThreads), 0, st, p)) != cudaSuccess) return e;
  if ((e = launch_pdl(layer_count_kernel, grid, dim3(kSelThreads), 0, st, p)) != cudaSuccess) return e;
  return launch_pdl(layer_write_kernel, grid, dim3(kSelThreads), 0, st, p);
}

cudaError_t launch_compact(const CompactParams& p, cudaStream_t st) {
  if (p.out_rows <= 0) return cudaSuccess;
  // about four waves of 8 resident CTAs per SM over all heads, at most one
  // CTA per kRowsPerBlock output rows
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorUnknown;
  const int units = p.B * p.Hkv;
  const int per_unit = std::max(1, 4 * 8 * sms / units);
  dim3 grid(std::min((p.out_rows + kRowsPerBlock - 1) / kRowsPerBlock, per_unit), units);
  return launch_pdl(compact_kernel, grid, dim3(kCompactThreads), 0, st, p);
}

}  // namespace dropkv
