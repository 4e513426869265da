// Pass 1 (window attention with split-K, then a merge of the splits) and pass 2
// (streaming per-token perturbation score) of the DropKV scoring path.
//
// Both passes stream 128-token K/V tiles of one KV head through TMA into
// 128-byte-swizzled shared memory and put the two small contractions on the
// tcgen05 tensor cores with fp32 accumulators in TMEM:
//   S^T [128 tokens x R rows] = K_tile . Q^T        (A = K, K-major; B = Q, K-major)
//   pass 1: O^T [128 dims x R] += V_tile^T . P^T     (A = V, MN-major; B = P, MN-major)
//   pass 2: AV^T [128 tokens x R] = V_tile . a^T     (A = V, K-major; B = a_hi, then a_lo)
// with one TMEM lane per token (or per head dimension for O).  Eight worker
// warps own the 128 lanes twice over (warps w and w + 4 read lane quarter w)
// and split the R window rows between them, so each worker thread owns one
// token and half of the rows and needs no cross-thread reduction on the hot
// path; a TMA warp and an MMA warp feed them through mbarrier rings.  Each
// pass runs one wave of CTAs shared out over the KV heads (floor(SMs / U) per
// head for one sequence, in proportion to the lengths for a ragged batch).
// Pass 1 splits a head's tiles statically over its CTAs (one partial state
// each, merged by merge_splits_kernel); pass 2's CTAs claim the head's tiles
// dynamically.  The SnapKV score kind runs the same kernels with K only
// (pass 1 keeps the softmax statistics, pass 2 sums p over the window).
//
// Method: "DropKV: Exact single-entry output-perturbation scoring", Core
// equation (p = softmax(Kq/sqrt d), a = sum_j p_j v_j, Delta_j = p_j/(1-p_j)
// (a - v_j), s_j = sum_t |Delta_j^(t)|^2), Algorithm 1 summary (GQA average,
// singular inputs rejected) and Code mapping (tail-aligned causality);
// "DropKV: Decoupling Residual-Output Perturbation ...", Appendix D (a
// FlashAttention-style pass for outputs and log-sum-exp, split-K partial
// states merged, then a second pass accumulating scores over key tiles without
// materialising the attention matrix).
#include <cuda_bf16.h>
#include <algorithm>
#include <cuda_runtime.h>

#include "dropkv_internal.cuh"
#include "sm103_ptx.cuh"

namespace dropkv {
namespace {

constexpr int kWorkerWarps = 8;          // warps w and w + 4 share TMEM lane quarter w and split the rows
constexpr int kWorkers = 32 * kWorkerWarps;
constexpr int kProducerWarp = 8;         // TMA producer
constexpr int kMmaWarp = 9;              // MMA issuer, TMEM owner
constexpr int kThreads = 320;
constexpr int kTileBytes = kTile * kDPad * 2;   // 32 KB: one K or V tile, two SW128 blocks
constexpr int kHalfTile = kTileBytes / 2;
constexpr uint32_t kBarWork = 1, kBarAux = 2;    // named barriers among the worker warps
// Lazy re-referencing of the running softmax maximum (log2 units): the
// exponentials of a CTA stay relative to one reference until some logit
// exceeds it by more than this, so e = 2^(y - ref) <= 2^24.
constexpr float kRescaleLog2 = 24.0f;
constexpr uint64_t kDrainNs = 20000000ull;   // 20 ms to drain copies after an abort

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Order-preserving map of floats to unsigned ints (for max reductions).
__device__ __forceinline__ uint32_t f2ord(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord2f(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------ grid sharing
// A pass grid of G = p.ctas CTAs (one wave) is shared out over the KV heads.
// With one sequence (or no lengths) every head gets p.even CTAs, known from
// the CTA index alone.  Otherwise the share follows the lengths: sequence b
// has T_b = ceil(n_b / kTile) tiles in each of its heads, and each of those
// heads gets
//   s_b = min(p.splits, T_b, 1 + floor((G - U) T_b / (Hkv sum_b' T_b')))
// CTAs: every head gets one, the rest go by length, and sum_u s_u <= G.  A
// length outside [w, n_max] counts as one tile (the head's one CTA flags it).
// Every lane of a warp computes the same result from the lengths alone, so
// all CTAs of a pass and the merge kernel agree on it.  The products fit in
// 32 bits: when G > U both G and U are below 256 (the host caps G there),
// T_b <= 2^24, and split bounds are at most kMaxSplits 2^24.
__device__ __forceinline__ int seq_len(const AttnParams& p, int b) { return p.lengths ? p.lengths[b] : p.n_max; }
__device__ __forceinline__ int seq_tiles(const AttnParams& p, int nb) {
  return (nb < p.w || nb > p.n_max) ? 1 : ceil_div(nb, kTile);
}
// Hkv times the sum over the sequences of T_b
__device__ __forceinline__ uint32_t total_tiles(const AttnParams& p) {
  uint32_t t = 0;
  for (int b = threadIdx.x & 31; b < p.B; b += 32) t += (uint32_t)seq_tiles(p, seq_len(p, b));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t * (uint32_t)p.Hkv;
}
__device__ __forceinline__ int seq_share(const AttnParams& p, int tiles, uint32_t tot) {
  const uint32_t extra = (uint32_t)(p.ctas - p.U);
  const int s = extra ? 1 + (int)(extra * (uint32_t)tiles / tot) : 1;
  return min(min(p.splits, tiles), s);
}

struct CtaWork {
  int unit;     // b * Hkv + h, or -1: a CTA left over, no work in this pass
  int split;    // 0 .. nsplit-1
  int nsplit;   // CTAs of this unit
  int nb;       // length of the unit's sequence
};

// Work of CTA `cta`: the units are laid out sequence by sequence, head by
// head, each with its s_b consecutive CTAs.  Warp-uniform.
__device__ CtaWork cta_work(const AttnParams& p, int cta) {
  CtaWork wk{-1, 0, 0, 0};
  if (p.even > 0) {
    if (cta >= p.U * p.even) return wk;
    if (p.even >= 8) {
      // many CTAs per head: heads interleaved over the grid (CTA c serves
      // head c mod U), so that each head's CTAs sit on SMs all over the chip
      // and pass 2's heads, each claiming from its own counter, finish together
      wk.split = cta / p.U;
      wk.unit = cta - wk.split * p.U;
    } else {
      wk.unit = cta / p.even;
      wk.split = cta - wk.unit * p.even;
    }
    wk.nsplit = p.even;
    wk.nb = seq_len(p, wk.unit / p.Hkv);
    return wk;
  }
  const int lane = threadIdx.x & 31;
  const uint32_t tot = total_tiles(p);
  int base = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    const int nb = b < p.B ? seq_len(p, b) : 0;
    const int s = b < p.B ? seq_share(p, seq_tiles(p, nb), tot) : 0;
    int incl = s * p.Hkv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    incl += base;
    const unsigned hit = __ballot_sync(0xffffffffu, b < p.B && cta < incl);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const int sb = __shfl_sync(0xffffffffu, s, src);
      const int start = __shfl_sync(0xffffffffu, incl, src) - sb * p.Hkv;
      wk.nb = __shfl_sync(0xffffffffu, nb, src);
      const int h = (cta - start) / sb;
      wk.unit = (b0 + src) * p.Hkv + h;
      wk.split = cta - start - h * sb;
      wk.nsplit = sb;
      break;
    }
    base = __shfl_sync(0xffffffffu, incl, 31);
  }
  return wk;
}

// Wait for a copy or MMA to land without honouring the abort flag (used only
// to drain work in flight before the CTA exits).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 26) && !mbar_try_wait(bar, parity); ++it)
    if (global_timer_ns() - t0 > kDrainNs) break;
}

// Stage `rows` x 128 bf16 of a row-major [rows_valid][ld] matrix into the
// K-major SW128 layout, zero-filling rows >= rows_valid and columns >= cols.
__device__ __forceinline__ void stage_rows_sw128(uint8_t* dst, const __nv_bfloat16* src, int rows, int rows_valid,
                                                 int ld, int cols, int tid, int nthr) {
  for (int idx = tid; idx < rows * 16; idx += nthr) {
    const int r = idx >> 4, c8 = idx & 15;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < rows_valid && c8 * 8 < cols) val = *reinterpret_cast<const uint4*>(src + (size_t)r * ld + c8 * 8);
    *reinterpret_cast<uint4*>(dst + sw128_offset(r, c8 * 8, rows)) = val;
  }
}

// Two fp32 values as bf16 hi parts plus bf16 lo parts (e = hi + lo to ~2^-17).
__device__ __forceinline__ void split_hi_lo(float e0, float e1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(e0, e1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(e0 - hf.x, e1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Max of two pairs of non-negative bf16 values (their bit patterns order as
// unsigned 16-bit integers).
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
  const __nv_bfloat162 m =
      __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&m);
}
// A pair of bf16 values times (f0, f1), rounded back to bf16.
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t a, float f0, float f1) {
  const __nv_bfloat162 h =
      __floats2bfloat162_rn(__uint_as_float(a << 16) * f0, __uint_as_float(a & 0xFFFF0000u) * f1);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Sum of squares of 8 packed bf16 values.
__device__ __forceinline__ float sumsq_bf16x8(const uint4 v, float acc) {
  const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float lo = __uint_as_float(w4[u] << 16), hi = __uint_as_float(w4[u] & 0xFFFF0000u);
    acc = fmaf(lo, lo, acc);
    acc = fmaf(hi, hi, acc);
  }
  return acc;
}

#ifdef DROPKV_TEST_HOOKS
// Test build only: the (unit, tile) whose K copy the prefill attention leaves
// out, so that the MMA issuer's bounded wait for it runs out and the kernel
// takes its timeout exit.  {-1, -1}: none.
__device__ int g_test_skip_pf_k[2] = {-1, -1};
#endif

// TMA producer of one ring: streams the tiles [t0, t0 + T) of one tensor into
// a ring of DEPTH 32 KB stages.  K and V rings are driven by different lanes
// of the producer warp, so each can run ahead of the consumers by its own depth.
// The first `start` tiles were issued already (during the CTA's set-up).
// HOOK: the prefill's K stream (the test build may leave one copy out).
template <int DEPTH, bool HOOK = false>
__device__ __forceinline__ void stream_ring(uint8_t* ring, uint64_t* full, uint64_t* empty, const CUtensorMap* map,
                                            int t0, int T, int unit, int start, volatile int* abort,
                                            uint32_t* status) {
  int issued = start;
  bool ok = true;
  for (int i = start; i < T; ++i) {
    const int s = i % DEPTH;
    if (i >= DEPTH && !mbar_wait(&empty[s], ((i / DEPTH) + 1) & 1, abort)) { ok = false; break; }
#ifdef DROPKV_TEST_HOOKS
    if (!HOOK || unit != g_test_skip_pf_k[0] || t0 + i != g_test_skip_pf_k[1])
#endif
    {
      mbar_arrive_expect_tx(&full[s], kTileBytes);
      tma_load_3d(ring + s * kTileBytes, map, &full[s], 0, (t0 + i) * kTile, unit);
      tma_load_3d(ring + s * kTileBytes + kHalfTile, map, &full[s], 64, (t0 + i) * kTile, unit);
    }
    ++issued;
  }
  if (!ok) {
    *abort = 1;
    atomicOr(status, DROPKV_FLAG_TIMEOUT);
    for (int i = max(0, issued - DEPTH); i < issued; ++i) mbar_drain(&full[i % DEPTH], (i / DEPTH) & 1);
  }
}

// ============================================================== pass 1
constexpr int kMaxStages = 6;   // ring stages of one tensor (mbarrier arrays)

// STATS: statistics only (no V): the V ring's stages go to K, keeping the
// bytes in flight per SM (V keeps one unused stage so the ring arithmetic holds).
template <int NR, bool STATS = false>
struct Pass1Cfg {
  static constexpr int HR = NR / 2;                 // rows per worker half
  static constexpr int KS0 = NR <= 16 ? 3 : 2;      // K ring depth (K is released right after S = K Q^T)
  static constexpr int VS0 = 3;                     // V ring depth (V is held until PV completes)
  static constexpr int KS = STATS ? KS0 + VS0 - 1 : KS0;
  static constexpr int VS = STATS ? 1 : VS0;
  // One P buffer: the workers write P(i) once PV(i-1) is done.  Measured on
  // GB300 at n = 128K, a second buffer made the pass slower (1.50 against
  // 1.42 us per tile per CTA), and deeper K or V rings gained nothing.
  static constexpr int PB = 1;
  static constexpr int kQBytes = NR * kDPad * 2;
  static constexpr int kPBytes = kTile * NR * 2;    // one of (hi, lo) of one P buffer
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + KS * kTileBytes;
  static constexpr int kOffQ = kOffV + VS * kTileBytes;
  static constexpr int kOffP = kOffQ + kQBytes;     // [buffer][hi, lo]
  static constexpr int kOffSmall = kOffP + 2 * PB * kPBytes;
  static constexpr uint32_t kTmemCols = (3 * NR <= 64) ? 64u : (3 * NR <= 128 ? 128u : 256u);
  static_assert(KS <= kMaxStages && VS <= kMaxStages, "ring depth");
};

struct Pass1Small {
  uint64_t kfull[kMaxStages], kempty[kMaxStages], vfull[kMaxStages], vempty[kMaxStages];
  uint64_t sfull[2], sempty[2], pfull[2], pempty[2], ofull, drain;
  uint32_t tmem_base;
  int abort;
  int pos[kMaxR];          // last key visible to row r (tail-aligned causality)
  float mref[kMaxR];       // exponent reference of row r (log2 units; live for NR = 64, else at the end)
  float mnew[kMaxR];       // staging of a new reference (NR = 64)
  float red[4][kMaxR];     // per-lane-quarter reduction scratch
  uint32_t rmax[4][kMaxR]; // per lane quarter: largest e of row r (bf16 bits of a non-negative value)
};

template <int NR, bool STATS>
constexpr int pass1_smem_bytes() {
  return Pass1Cfg<NR, STATS>::kOffSmall + (int)sizeof(Pass1Small) + 1024;
}

// Merge of the split-K partial states (its own small kernel: it sits on the
// critical path, so it is spread over many CTAs with all loads in flight).
//   m = max_s m_s;  L = sum_s l_s 2^(m_s - m);  a = sum_s O_s 2^(m_s - m) / L.
// CTA (row group, KV head): warp w < 4 takes row r = 4 * group + w.  Lane c
// holds the (m, l, largest e) of splits c, c + 32, ... and float4 column c of
// every split's O, all requested in one round trip.  Writes a, m, L and the
// exported log-sum-exp.
//
// Shift of the scoring basis: the partial output of row 0 over the split that
// holds tile 0 (a weighted average of values, read in the same round trip by
// every warp), rounded to bf16, is the head's shift c when |c|^2 > 2 d (the
// values share an offset large against their spread), else c = 0.  Each row
// is written as a' = a - c, split into bf16 hi + lo parts (pass 2's A.V^T
// operand; rows past R are zero), with K = |a'|^2 + 2 a'.c, so that pass 2
// evaluates |a - v|^2 = K - 2 a'.v + |v - c|^2 without the cancellation of
// |a|^2 - 2 a.v + |v|^2 when |v| is far above |a - v|.
//
// A row whose largest probability p* = e* / L reaches kDomP (e* = the largest
// e of any split, weighted like its l) is dominated: the merge records the
// split s* that holds that key (unique, since p* > 1/2) and the (O, L) of
// every other split -- sums whose terms do not contain the dominant key, from
// which pass 2 rebuilds the output without that key with no cancellation.
// Each split's largest e comes from the bf16 hi parts of pass 1's P operand:
// good to 2^-9, which only blurs the threshold; pass 2 uses the key's own e.
constexpr int kMergeRows = 4;                 // rows per CTA (one warp each)
constexpr int kMergeThreads = 32 * kMergeRows;
constexpr int kMergeSplitRegs = kMaxSplits / 32;
static_assert(kMergeSplitRegs * 32 == kMaxSplits, "split states are held 32 per register slot");

__global__ void __launch_bounds__(kMergeThreads) merge_splits_kernel(const AttnParams p) {
  // the O column of up to 32 splits per row (warp), [warp][split][lane],
  // staged with cp.async: in flight with the statistics' loads, and the
  // reduction below runs as a short loop (this kernel's code is fetched cold)
  extern __shared__ float4 mo_s[];
  __shared__ float wts_s[kMergeRows][32];
  __shared__ float wex_s[kMergeRows][32];       // the same weights without split s* (dominated rows)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.y, r = blockIdx.x * kMergeRows + warp;
  const int b = unit / p.Hkv;
  // caller inputs, read before the wait: the length and pass 1's split count
  const int nb = seq_len(p, b);
  const int S = p.part_splits > 0 ? p.part_splits
                : (p.even > 0 ? p.even : seq_share(p, seq_tiles(p, nb), total_tiles(p)));
  grid_dep_wait();                                // the partials come from pass 1
  // Pass 2's CTAs may be scheduled now when this grid fits in one wave (their
  // start-up then overlaps the merge); a larger merge grid triggers them only
  // as its CTAs exit, so that they do not take the SM slots its later CTAs
  // wait for.
  if (gridDim.x * gridDim.y <= (unsigned)p.ctas) grid_dep_launch();
  if (blockIdx.x == 0 && threadIdx.x == 0) p.tile_ctr[unit] = 0;   // pass 2 claims its tiles from 0
  if (nb < p.w || nb > p.n_max) return;          // flagged by pass 1 (the whole CTA leaves)
  const int R = p.R, d = p.d, D4 = d >> 2;
  const bool stats_only = p.kind == kKindSnapKV;   // no O partials were written
  const bool live = r < R;
  const size_t ro = (size_t)unit * R + r;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  float M = -INFINITY, L = 0.f, Lx = 0.f;
  bool dom = false;
  int sstar = -1;
  // the shift's source: row 0 of the split that holds tile 0 (split
  // ceil(S / T) - 1 when a head has fewer tiles T than splits S)
  float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c = c0;
  float c0l = 0.f;
  if (!stats_only) {
    const int T = ceil_div(nb, kTile);
    const int s0 = T >= S ? 0 : ceil_div(S, T) - 1;
    c0l = __ldcg(p.part_ml + ((size_t)unit * p.splits + s0) * R * 4 + 1);
    if (lane < D4) c0 = __ldcg(reinterpret_cast<const float4*>(p.part_o + ((size_t)unit * p.splits + s0) * R * d) + lane);
  }
  if (live) {
    const float4* ml = reinterpret_cast<const float4*>(p.part_ml) + (size_t)unit * p.splits * R;
    const float4* po4 = reinterpret_cast<const float4*>(p.part_o + (size_t)unit * p.splits * R * d);
    const size_t split_stride = (size_t)R * D4;
    // one round trip: the (m, l, largest e) of every split and the O column
    // of the first 32 splits are all requested before any is used (the O
    // partial of a split without visible keys is never written; its weight is
    // 0 and it is dropped by a select, not a multiply, so whatever it holds
    // cannot leak in)
    float4 v[kMergeSplitRegs];
#pragma unroll
    for (int q = 0; q < kMergeSplitRegs; ++q) {
      const int s = q * 32 + lane;
      v[q] = (s < S) ? __ldcg(ml + (size_t)s * R + r) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
    }
    const int CH = min(32, p.splits);            // splits staged per round (the launch sized mo_s for it)
    float4* mo = mo_s + (size_t)warp * CH * 32;
    auto stage = [&](int q) {
      if (stats_only || lane >= D4) return;
      const int n = min(CH, S - q * CH);
#pragma unroll 1
      for (int u = 0; u < n; ++u)
        cp_async_cg16(mo + u * 32 + lane, po4 + (size_t)(q * CH + u) * split_stride + (size_t)r * D4 + lane);
    };
    stage(0);
#pragma unroll
    for (int q = 0; q < kMergeSplitRegs; ++q)
      if (v[q].y > 0.f) M = fmaxf(M, v[q].x);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    float wgt[kMergeSplitRegs];
    float E = 0.f;                 // the largest e of any split, in the merged reference
#pragma unroll
    for (int q = 0; q < kMergeSplitRegs; ++q) {
      wgt[q] = (v[q].y > 0.f) ? exp2f(v[q].x - M) : 0.f;
      L = fmaf(v[q].y, wgt[q], L);
      E = fmaxf(E, v[q].z * wgt[q]);
    }
    L = warp_sum(L);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) E = fmaxf(E, __shfl_xor_sync(0xffffffffu, E, o2));
    if (!stats_only) {
      // c = bf16(the source's output) when it is large (|c|^2 > 2 d), else 0;
      // the same in every warp of the head (its loads were issued first)
      const float inv0 = c0l > 0.f ? 1.0f / c0l : 0.f;
      const __nv_bfloat162 c01 = __floats2bfloat162_rn(c0.x * inv0, c0.y * inv0);
      const __nv_bfloat162 c23 = __floats2bfloat162_rn(c0.z * inv0, c0.w * inv0);
      const float2 f01 = __bfloat1622float2(c01), f23 = __bfloat1622float2(c23);
      const float cc = warp_sum(f01.x * f01.x + f01.y * f01.y + f23.x * f23.x + f23.y * f23.y);
      const bool shift = cc > 2.0f * (float)d;    // also false for a non-finite source
      c = shift ? make_float4(f01.x, f01.y, f23.x, f23.y) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (blockIdx.x == 0 && warp == 0) {
        reinterpret_cast<float4*>(p.cvec + (size_t)unit * kDPad)[lane] = c;
        if (lane == 0) p.cflag[unit] = shift ? 1 : 0;
      }
    }
    dom = !stats_only && E >= kDomP * L;        // the same in every lane
    float wex[kMergeSplitRegs];
    if (dom) {
      int first = 0x7fffffff;
#pragma unroll
      for (int q = 0; q < kMergeSplitRegs; ++q)
        if (v[q].y > 0.f && v[q].z * wgt[q] == E) first = min(first, q * 32 + lane);
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o2));
      sstar = first;
#pragma unroll
      for (int q = 0; q < kMergeSplitRegs; ++q) {
        wex[q] = (q * 32 + lane == sstar) ? 0.f : wgt[q];
        Lx = fmaf(v[q].y, wex[q], Lx);
      }
      Lx = warp_sum(Lx);
    }
    if (!stats_only) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), acx = make_float4(0.f, 0.f, 0.f, 0.f);
      // splits in order, CH at a time (their weights through wts_s / wex_s,
      // 32 per register slot); a split without visible keys has weight 0 and
      // is dropped by a select, not a multiply, so whatever its O holds
      // cannot leak in
      for (int q = 0; q * CH < S; ++q) {
        if (q > 0) stage(q);
        cp_async_wait_all();
        const int n = min(CH, S - q * CH);
#pragma unroll 1
        for (int u = 0; u < n; ++u) {
          const int s = q * CH + u;                 // split index
          if ((s & 31) == 0) {                      // the next 32 splits' weights
            const int qi = s >> 5;
            float w0 = wgt[0], x0 = dom ? wex[0] : 0.f;
#pragma unroll
            for (int k = 1; k < kMergeSplitRegs; ++k)
              if (k == qi) {
                w0 = wgt[k];
                if (dom) x0 = wex[k];
              }
            __syncwarp();
            wts_s[warp][lane] = w0;
            wex_s[warp][lane] = x0;
            __syncwarp();
          }
          const float wu = wts_s[warp][s & 31];
          const float wx = wex_s[warp][s & 31];
          const float4 ov = mo[u * 32 + lane];
          if (wu != 0.f) {
            acc.x = fmaf(ov.x, wu, acc.x);
            acc.y = fmaf(ov.y, wu, acc.y);
            acc.z = fmaf(ov.z, wu, acc.z);
            acc.w = fmaf(ov.w, wu, acc.w);
          }
          if (dom && wx != 0.f) {
            acx.x = fmaf(ov.x, wx, acx.x);
            acx.y = fmaf(ov.y, wx, acx.y);
            acx.z = fmaf(ov.z, wx, acx.z);
            acx.w = fmaf(ov.w, wx, acx.w);
          }
        }
        __syncwarp();                                // the next round overwrites mo
      }
      const float inv = 1.0f / L;
      a = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      if (lane >= D4) a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane < D4) reinterpret_cast<float4*>(p.a + ro * d)[lane] = a;
      if (dom && lane < D4) reinterpret_cast<float4*>(p.dom_o + ro * d)[lane] = acx;
    }
    if (lane == 0) {
      p.m2[ro] = M;
      p.l[ro] = L;
      // exported: log-sum-exp of the natural-unit logits, log(L) + m ln 2
      p.m[ro] = (M + log2f(L)) * 0.69314718055994531f;
      if (!stats_only) {
        p.dom_s[ro] = sstar;
        p.dom_l[ro] = Lx;
      }
    }
  }
  if (stats_only) {
    if (live && lane == 0 && (!(L > 0.f) || !isfinite(L)))
      atomicOr(p.status, DROPKV_FLAG_NONFINITE | DROPKV_FLAG_NONFINITE_STATS);
    return;
  }
  __nv_bfloat16* ahl = p.ahl + (size_t)unit * 2 * kMaxR * kDPad;
  if (!live) {
    // padding rows of the MMA operand: zero (32 lanes x 4 columns = 128)
    reinterpret_cast<uint2*>(ahl + (size_t)r * kDPad)[lane] = make_uint2(0u, 0u);
    reinterpret_cast<uint2*>(ahl + (size_t)(kMaxR + r) * kDPad)[lane] = make_uint2(0u, 0u);
    return;
  }
  const float4 ap = make_float4(a.x - c.x, a.y - c.y, a.z - c.z, a.w - c.w);
  // K = |a'|^2 + 2 a'.c
  const float K = warp_sum(ap.x * (ap.x + 2.f * c.x) + ap.y * (ap.y + 2.f * c.y) + ap.z * (ap.z + 2.f * c.z) +
                           ap.w * (ap.w + 2.f * c.w));
  uint32_t h01, l01, h23, l23;
  split_hi_lo(ap.x, ap.y, h01, l01);
  split_hi_lo(ap.z, ap.w, h23, l23);
  reinterpret_cast<uint2*>(ahl + (size_t)r * kDPad)[lane] = make_uint2(h01, h23);
  reinterpret_cast<uint2*>(ahl + (size_t)(kMaxR + r) * kDPad)[lane] = make_uint2(l01, l23);
  if (lane == 0) {
    p.aa[ro] = K;
    if (!(L > 0.f) || !isfinite(L) || !isfinite(K))
      atomicOr(p.status, DROPKV_FLAG_NONFINITE | DROPKV_FLAG_NONFINITE_STATS);
  }
}

// STATS: the softmax statistics (m, l) only -- no V, no P V^T, no O partial
// (the SnapKV score needs the normaliser of every window row, not a).
template <int NR, bool STATS>
__global__ void __launch_bounds__(kThreads, 1)
    window_attention_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                            const AttnParams p) {
  using C = Pass1Cfg<NR, STATS>;
  constexpr int HR = C::HR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sK = sm + C::kOffK;
  uint8_t* sV = sm + C::kOffV;
  uint8_t* sQ = sm + C::kOffQ;
  uint8_t* sP = sm + C::kOffP;
  Pass1Small& S = *reinterpret_cast<Pass1Small*>(sm + C::kOffSmall);

  // The lengths, Q, K and V are the caller's, and the kernel before this one
  // (a previous call's compaction, for one) may still be writing them.
  grid_dep_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const CtaWork wk = cta_work(p, blockIdx.x);
  if (wk.unit < 0) return;                  // left over: no work in this pass
  const int split = wk.split, unit = wk.unit, nb = wk.nb;
  // an even static split of the unit's tiles: floor or ceil of ntiles / nsplit each
  const int ntiles = ceil_div(nb, kTile);
  const int t0 = (int)((uint32_t)split * (uint32_t)ntiles / (uint32_t)wk.nsplit);
  const int t1 = (int)((uint32_t)(split + 1) * (uint32_t)ntiles / (uint32_t)wk.nsplit);
  const int b = unit / p.Hkv, h = unit - b * p.Hkv;
  if (nb < p.w || nb > p.n_max) {           // invalid length: the unit is skipped
    if (tid == 0 && split == 0 && h == 0) atomicOr(p.status, DROPKV_FLAG_BAD_LENGTH);
    return;
  }
  const int R = p.R;
  const int T = max(0, t1 - t0);

  // Set-up.  The producer lane sets up the rings' barriers itself and issues
  // the first stages of both rings at once, so the first tiles are in flight
  // while the other warps set up.
  int k_issued = 0, v_issued = 0;
  if (warp == kProducerWarp && lane == 0) {
    for (int i = 0; i < C::KS; ++i) { mbar_init(&S.kfull[i], 1); mbar_init(&S.kempty[i], 1); }
    for (int i = 0; i < C::VS; ++i) { mbar_init(&S.vfull[i], 1); mbar_init(&S.vempty[i], 1); }
    S.abort = 0;
    fence_mbar_init();
    if (T > 0) {
      tma_prefetch_desc(&tmk);
      if (!STATS) tma_prefetch_desc(&tmv);
      k_issued = min(T, C::KS);
      for (int i = 0; i < k_issued; ++i) {
        mbar_arrive_expect_tx(&S.kfull[i], kTileBytes);
        tma_load_3d(sK + i * kTileBytes, &tmk, &S.kfull[i], 0, (t0 + i) * kTile, unit);
        tma_load_3d(sK + i * kTileBytes + kHalfTile, &tmk, &S.kfull[i], 64, (t0 + i) * kTile, unit);
      }
      if (!STATS) {
        v_issued = min(T, C::VS);
        for (int i = 0; i < v_issued; ++i) {
          mbar_arrive_expect_tx(&S.vfull[i], kTileBytes);
          tma_load_3d(sV + i * kTileBytes, &tmv, &S.vfull[i], 0, (t0 + i) * kTile, unit);
          tma_load_3d(sV + i * kTileBytes + kHalfTile, &tmv, &S.vfull[i], 64, (t0 + i) * kTile, unit);
        }
      }
    }
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) { mbar_init(&S.sfull[i], 1); mbar_init(&S.sempty[i], kWorkerWarps); }
    for (int i = 0; i < C::PB; ++i) { mbar_init(&S.pfull[i], kWorkerWarps); mbar_init(&S.pempty[i], 1); }
    mbar_init(&S.ofull, 1);
    mbar_init(&S.drain, 1);
    fence_mbar_init();
  }
  if (tid < kMaxR) {
    S.pos[tid] = (tid < R) ? nb - p.w + (tid % p.w) : -1;
    S.mref[tid] = -INFINITY;
  }
  if (T > 0) {
    if (warp == kMmaWarp) tmem_alloc(&S.tmem_base, C::kTmemCols);
    if (tid < kWorkers) {
      const __nv_bfloat16* qsrc = p.q + ((size_t)b * p.Hq + (size_t)h * p.g) * p.w * p.d;
      stage_rows_sw128(sQ, qsrc, NR, R, p.d, p.d, tid, kWorkers);
      fence_proxy_async_smem();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const uint32_t tS = tmem, tO = tmem + 2 * NR;    // S buffers at [0, 2NR), O at [2NR, 3NR)
  bool failed = false;
  // Streaming reads only the caller's inputs, so the next kernel may be
  // scheduled now; the writes of the partial states come after grid_dep_wait().
  grid_dep_launch();

  if (T > 0 && warp == kProducerWarp) {
    // ---------------------------------------------------- TMA producer: lane 0 K, lane 1 V
    // lane 0 issued the first stages of both rings during the set-up
    const int kis = __shfl_sync(0xffffffffu, k_issued, 0), vis = __shfl_sync(0xffffffffu, v_issued, 0);
    if (lane == 0) stream_ring<C::KS>(sK, S.kfull, S.kempty, &tmk, t0, T, unit, kis, &S.abort, p.status);
    else if (lane == 1 && !STATS) stream_ring<C::VS>(sV, S.vfull, S.vempty, &tmv, t0, T, unit, vis, &S.abort, p.status);
    __syncwarp();
  } else if (T > 0 && warp == kMmaWarp) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idS = umma_idesc_bf16(128, NR, 0, 0);
      const uint32_t idO = umma_idesc_bf16(128, NR, 1, 1);
      const uint32_t qaddr = smem_addr(sQ);
      bool ok = true;
      auto issue_S = [&](int i) -> bool {
        const int ks = i % C::KS, sb = i & 1;
        if (!mbar_wait(&S.kfull[ks], (i / C::KS) & 1, &S.abort)) return false;
        if (i >= 2 && !mbar_wait(&S.sempty[sb], ((i >> 1) + 1) & 1, &S.abort)) return false;
        tc_fence_after();
        const uint32_t kb = smem_addr(sK + ks * kTileBytes);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_bf16(tS + sb * NR, desc_kmajor_sw128(kb, kTile, s), desc_kmajor_sw128(qaddr, NR, s), idS, s > 0);
        umma_commit(&S.sfull[sb]);
        umma_commit(&S.kempty[ks]);
        return true;
      };
      ok = issue_S(0);
      for (int i = 0; ok && i < T; ++i) {
        if (i + 1 < T && !(ok = issue_S(i + 1))) break;
        if (STATS) continue;
        const int pb = i % C::PB, vs = i % C::VS;
        if (!mbar_wait(&S.pfull[pb], (i / C::PB) & 1, &S.abort)) { ok = false; break; }
        if (!mbar_wait(&S.vfull[vs], (i / C::VS) & 1, &S.abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vb = smem_addr(sV + vs * kTileBytes);
        const uint32_t phi = smem_addr(sP + (pb * 2 + 0) * C::kPBytes);
        const uint32_t plo = smem_addr(sP + (pb * 2 + 1) * C::kPBytes);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_bf16(tO, desc_mnmajor_sw128(vb, kTile, s), desc_mnmajor_interleave(phi, NR, s), idO, (i > 0 || s > 0));
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_bf16(tO, desc_mnmajor_sw128(vb, kTile, s), desc_mnmajor_interleave(plo, NR, s), idO, 1);
        umma_commit(&S.vempty[vs]);
        umma_commit(&S.pempty[pb]);
        umma_commit(&S.ofull);
      }
      if (!ok) {
        failed = true;
        S.abort = 1;
        atomicOr(p.status, DROPKV_FLAG_TIMEOUT);
      }
      // make sure no MMA is still writing TMEM before it is released
      umma_commit(&S.drain);
      mbar_drain(&S.drain, 0);
    }
    __syncwarp();
  } else if (T > 0 && warp < kWorkerWarps) {
    // ---------------------------------------------------- softmax workers
    // Thread (quarter wq, half) owns token wq*32 + lane of each tile and rows
    // [r0, r0 + HR) of the window.
    const int wq = warp & 3, half = warp >> 2;
    const int tok = wq * 32 + lane;
    const int r0 = half * HR;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    uint32_t rowmask = 0;
#pragma unroll
    for (int r = 0; r < HR; ++r) rowmask |= (uint32_t)(r0 + r < R) << r;
    const float scale = p.scale_log2;
    const int all_see = nb - p.w;            // keys j <= all_see are visible to every row
    // The exponent reference of a row is the same in every thread.  For
    // NR <= 32 each thread keeps it in registers; for NR = 64 it stays in
    // shared memory (S.mref), which keeps the 32-row arrays of a thread within
    // the register budget of ten warps.
    constexpr bool kRefSmem = NR > 32;
    float lsum[HR], mr[kRefSmem ? 1 : HR];
    // Largest e of each row pair (r0 + 2q, r0 + 2q + 1), kept as the bf16 hi
    // parts the P operand is built from (one max per pair and token): the
    // merge finds from it the split that holds a row's largest probability
    // and whether that key dominates the row.
    uint32_t emax2[STATS ? 1 : HR / 2];
#pragma unroll
    for (int q = 0; q < (STATS ? 1 : HR / 2); ++q) emax2[q] = 0u;
#pragma unroll
    for (int r = 0; r < HR; ++r) lsum[r] = 0.f;
#pragma unroll
    for (int r = 0; r < (kRefSmem ? 1 : HR); ++r) mr[r] = -INFINITY;
    auto ref = [&](int r) -> float {
      if constexpr (kRefSmem) return S.mref[r0 + r];
      else return mr[r];
    };
    for (int i = 0; i < T; ++i) {
      const int tile0 = (t0 + i) * kTile, sb = i & 1, vs = i % C::VS, pb = i % C::PB;
      const int j = tile0 + tok;
      const bool full = tile0 + kTile - 1 <= all_see;
      const bool tail = tile0 + kTile > nb;       // tile holds slots past the sequence
      bool ok = __all_sync(0xffffffffu, mbar_wait(&S.sfull[sb], (i >> 1) & 1, &S.abort));
      float sraw[HR];
      if (ok) {
        tc_fence_after();
        tmem_ld_cols<HR>(tS + lane_base + sb * NR + r0, sraw);
        tmem_wait_ld();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.sempty[sb]);

      uint32_t vis = rowmask;
      if (!full) {
        uint32_t v = 0;
        if (j < nb) {
#pragma unroll
          for (int r = 0; r < HR; ++r) v |= (uint32_t)(j <= S.pos[r0 + r]) << r;
        }
        vis &= v;
      }
      bool need = false;
#pragma unroll
      for (int r = 0; r < HR; ++r) need |= ((vis >> r) & 1u) && fmaf(sraw[r], scale, -ref(r)) > kRescaleLog2;
      // this tile's P buffer must be free (PV of tile i - PB done); the tail tile's V must have landed
      if (!STATS && ok && i >= C::PB) ok = mbar_wait(&S.pempty[pb], ((i / C::PB) + 1) & 1, &S.abort);
      if (!STATS && ok && tail) ok = mbar_wait(&S.vfull[vs], (i / C::VS) & 1, &S.abort);
      ok = __all_sync(0xffffffffu, ok);
      // one barrier per tile in the common case: it carries both "some wait
      // failed" and "some logit outgrew its reference"
      if (named_bar_or(kBarWork, kWorkers, !ok || need)) {
        if (named_bar_or(kBarAux, kWorkers, !ok)) { failed = true; break; }
        // new reference = max(old reference, this tile's max) per row
#pragma unroll
        for (int r = 0; r < HR; ++r) {
          const float v = ((vis >> r) & 1u) ? sraw[r] * scale : -INFINITY;
          const uint32_t u = __reduce_max_sync(0xffffffffu, f2ord(v));
          if (lane == 0) S.red[wq][r0 + r] = ord2f(u);
        }
        named_bar(kBarAux, kWorkers);
        float factor[HR];
#pragma unroll
        for (int r = 0; r < HR; ++r) {
          const int rr = r0 + r;
          const float old = ref(r);
          const float nm = fmaxf(fmaxf(fmaxf(S.red[0][rr], S.red[1][rr]), fmaxf(S.red[2][rr], S.red[3][rr])), old);
          factor[r] = (old == -INFINITY) ? 0.f : ex2_approx(old - nm);
          lsum[r] *= factor[r];
          if (!STATS && (r & 1)) emax2[r >> 1] = scale_bf16x2(emax2[r >> 1], factor[r - 1], factor[r]);
          if constexpr (kRefSmem) {
            if (wq == 0 && lane == 0) S.mnew[rr] = nm;
          } else {
            mr[r] = nm;
          }
        }
        if constexpr (kRefSmem) {
          // every worker has read the old references: publish the new ones
          named_bar(kBarAux, kWorkers);
          if (wq == 0 && lane == 0)
            for (int r = 0; r < HR; ++r) S.mref[r0 + r] = S.mnew[r0 + r];
          named_bar(kBarAux, kWorkers);
        }
        if (!STATS && i > 0) {
          // rescale the accumulated O (lane = head dimension) once PV of tile i-1 is
          // done; PV(i-2) is known complete (pempty), so ofull is at most one phase
          // behind and the parity wait is unambiguous
          bool okw = mbar_wait(&S.ofull, (i - 1) & 1, &S.abort);
          okw = __all_sync(0xffffffffu, okw);
          if (named_bar_or(kBarAux, kWorkers, !okw)) { failed = true; break; }
          tc_fence_after();
          float o[HR];
          tmem_ld_cols<HR>(tO + lane_base + r0, o);
          tmem_wait_ld();
#pragma unroll
          for (int r = 0; r < HR; ++r) o[r] *= factor[r];
          tmem_st_cols<HR>(tO + lane_base + r0, o);
          tmem_wait_st();
          tc_fence_before();
        }
      }
      if (STATS) {
        // the normaliser only
#pragma unroll
        for (int r = 0; r < HR; ++r)
          if ((vis >> r) & 1u) lsum[r] += ex2_approx(fmaf(sraw[r], scale, -ref(r)));
        continue;
      }
      // exponentials relative to the row reference, split into bf16 hi + lo
      uint8_t* phi = sP + (pb * 2 + 0) * C::kPBytes;
      uint8_t* plo = sP + (pb * 2 + 1) * C::kPBytes;
#pragma unroll
      for (int c8 = 0; c8 < HR / 8; ++c8) {
        uint32_t hp[4], lp[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = c8 * 8 + 2 * q;
          const float e0 = ((vis >> r) & 1u) ? ex2_approx(fmaf(sraw[r], scale, -ref(r))) : 0.f;
          const float e1 = ((vis >> (r + 1)) & 1u) ? ex2_approx(fmaf(sraw[r + 1], scale, -ref(r + 1))) : 0.f;
          lsum[r] += e0;
          lsum[r + 1] += e1;
          split_hi_lo(e0, e1, hp[q], lp[q]);
          emax2[c8 * 4 + q] = max_bf16x2(emax2[c8 * 4 + q], hp[q]);
        }
        const uint32_t off = interleave_mn_offset(tok, r0 + c8 * 8, NR);
        *reinterpret_cast<uint4*>(phi + off) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
        *reinterpret_cast<uint4*>(plo + off) = make_uint4(lp[0], lp[1], lp[2], lp[3]);
      }
      if (tail && half == 0 && j >= nb) {
        // slots past the sequence may hold anything (NaN): zero their V rows
        // so that 0 * NaN never reaches the PV accumulator
        uint8_t* vrow = sV + vs * kTileBytes + tok * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vrow + kHalfTile + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pfull[pb]);
    }
    // ------------------------------------------------ partial state of this split
    // The MMA warp commits `drain` once, after its last MMA: a single-phase
    // wait.  (A parity wait on the per-tile `ofull` barrier would be ambiguous
    // here, since up to two PV commits may still be outstanding.)
    bool okw = true;
    if (!failed) okw = mbar_wait(&S.drain, 0, &S.abort);
    okw = __all_sync(0xffffffffu, okw);
    if (named_bar_or(kBarWork, kWorkers, failed || !okw)) failed = true;
    const size_t part = (size_t)unit * p.splits + split;
    if (!STATS && !failed) {
      tc_fence_after();
      float o[HR];
      tmem_ld_cols<HR>(tO + lane_base + r0, o);
      tmem_wait_ld();
      float* po = p.part_o + part * R * p.d;
#pragma unroll
      for (int r = 0; r < HR; ++r)
        if (r0 + r < R && tok < p.d) po[(size_t)(r0 + r) * p.d + tok] = o[r];
      tc_fence_before();
    }
#pragma unroll
    for (int r = 0; r < HR; ++r) {
      const float v = warp_sum(lsum[r]);
      if (lane == 0) S.red[wq][r0 + r] = v;
    }
    if constexpr (!STATS) {
#pragma unroll
      for (int q = 0; q < HR / 2; ++q) {
        const uint32_t lo = __reduce_max_sync(0xffffffffu, emax2[q] & 0xFFFFu);
        const uint32_t hi = __reduce_max_sync(0xffffffffu, emax2[q] >> 16);
        if (lane == 0) {
          S.rmax[wq][r0 + 2 * q] = lo;
          S.rmax[wq][r0 + 2 * q + 1] = hi;
        }
      }
    }
    if constexpr (!kRefSmem) {
      if (wq == 0 && lane == 0) {
#pragma unroll
        for (int r = 0; r < HR; ++r) S.mref[r0 + r] = mr[r];
      }
    }
    named_bar(kBarAux, kWorkers);
    if (tid < R) {
      // (reference, normaliser, largest e relative to the reference (bf16), unused)
      const uint32_t mx = STATS ? 0u : max(max(S.rmax[0][tid], S.rmax[1][tid]), max(S.rmax[2][tid], S.rmax[3][tid]));
      reinterpret_cast<float4*>(p.part_ml)[part * R + tid] =
          make_float4(S.mref[tid], failed ? 0.f : (S.red[0][tid] + S.red[1][tid]) + (S.red[2][tid] + S.red[3][tid]),
                      __uint_as_float(mx << 16), 0.f);
    }
  }

  if (T == 0) {
    // empty split (past the end of a shorter sequence): publish an empty state
    const size_t part = (size_t)unit * p.splits + split;
    for (int idx = tid; idx < R; idx += kThreads)
      reinterpret_cast<float4*>(p.part_ml)[part * R + idx] = make_float4(-INFINITY, 0.f, 0.f, 0.f);
  }

  tc_fence_before();
  __syncthreads();
  if (T > 0 && warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  // the partial states are merged by merge_splits_kernel
}

// ============================================================== pass 2
// Score of every token from the merged statistics of pass 1:
//   s_j = (1/g) sum_r r_r^2 |a_r - v_j|^2,   r_r = e / (L_r - e) = p / (1 - p),
// with |a_r - v_j|^2 evaluated in a basis shifted by c, the head's mean window
// output rounded to bf16:  K_r - 2 a'_r.v_j + |v_j - c|^2,  a' = a - c,
// K_r = |a'_r|^2 + 2 a'_r.c.  The products a'_r.v_j run on the tensor cores
// (a' split into bf16 hi + lo), |v_j - c|^2 is summed directly from the staged
// tile, and the shift keeps the expanded form accurate when the values share
// a large common offset (|v|^2 far above |a - v|^2).
//
// Mode of a CTA (chosen by the producer once the merge is done):
//  - dynamic: no row of the unit is dominated; the unit's CTAs claim its
//    tiles one at a time from a counter (the merge clears it).
//  - static: some row of the unit is dominated; every CTA of the unit takes
//    the tiles pass 1's split of the same index read, so the key a dominated
//    row hinges on is met by the CTA whose split the merge named.
//  - dominant: that CTA.  It leaves the dominant (row, key) pairs out of the
//    scores, accumulates O_rest^T += V^T P^T over its tiles with P = e of
//    every other visible key (tensor cores, a third TMEM accumulator, P staged
//    as in pass 1, one tile behind the scores), and at the end forms the window
//    output without the dominant key, a_rest = (O_other + O_rest) / (L_other +
//    L_rest), from sums that never contained that key, and adds the key's
//    exact term p*^2 |a_rest - v*|^2 (Delta = p / (1 - p) (a - v*) equals
//    p (a_rest - v*)) to its score.  When L_rest <= 2^-53 e*, p* rounds to 1
//    in double precision: the input is singular and the slot gets +inf.
enum : int { kModeDynamic = 0, kModeStatic = 1, kModeDominant = 2 };

// SNAP: K only; the V ring's shared memory goes to K.  Its barriers and tile
// indices stay (the workers learn each tile's index through the V slots), as
// deep as the K ring but with no data behind them.
template <int NR, bool SNAP = false>
struct Pass2Cfg {
  static constexpr int HR = NR / 2;
  static constexpr int KS0 = 2;                     // K is released right after S = K Q^T
  static constexpr int VS0 = NR <= 32 ? 4 : 3;      // V is held until A.V^T and |v - c|^2 are done
  static constexpr int KS = SNAP ? KS0 + VS0 : KS0;
  static constexpr int VS = SNAP ? KS : VS0;        // V slots (tile indices; data only without SNAP)
  static constexpr int kVStages = SNAP ? 0 : VS;    // V ring stages in shared memory
  static constexpr int kQBytes = NR * kDPad * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + KS * kTileBytes;
  static constexpr int kOffQ = kOffV + kVStages * kTileBytes;   // end of the ring region
  static constexpr int kOffAhi = kOffQ + kQBytes;
  static constexpr int kOffAlo = kOffAhi + kQBytes;
  static constexpr int kOffSmall = kOffAlo + kQBytes;
  // S and A.V^T double-buffered, then O_rest (dominant mode)
  static constexpr uint32_t kCols = SNAP ? 4 * NR : 5 * NR;
  static constexpr uint32_t kTmemCols = kCols <= 64 ? 64u : kCols <= 128 ? 128u : kCols <= 256 ? 256u : 512u;
  static_assert(KS <= kMaxStages && VS <= kMaxStages, "ring depth");
};

// Ring of the dominant mode: the same K ring and V stage addresses, a
// shallower V ring, and one P buffer (bf16 hi, then lo) for O_rest after it.
// (One copy of the producer and MMA code serves both modes.)
template <int NR>
struct Pass2Dom {
  static constexpr int VS = NR <= 32 ? 3 : 2;
  static constexpr int kPBytes = kTile * NR * 2;
  static constexpr int kOffP = Pass2Cfg<NR, false>::kOffV + VS * kTileBytes;
  static_assert(Pass2Cfg<NR, false>::KS == 2, "both modes share the K ring");
  static_assert(kOffP + 2 * kPBytes <= Pass2Cfg<NR, false>::kOffQ, "dominant ring exceeds the ring region");
};

struct Pass2Small {
  uint64_t kfull[kMaxStages], kempty[kMaxStages], vfull[kMaxStages], vempty[kMaxStages];
  int ktile[kMaxStages], vtile[kMaxStages];   // tile held by each ring slot (-1: no more tiles)
  uint64_t accfull[2], accempty[2], drain, aready, pfull, pempty;
  uint32_t tmem_base;
  int abort;
  int mode;                  // kMode*: written by the producer before it fills the first slot
  float4 pml[kMaxR / 2];     // per row pair (r, r + 1), r even: (-m_r, -m_r+1, L_r, L_r+1), m in log2 units
  float2 pk[kMaxR / 2];      // (K_r, K_r+1), K = |a'|^2 + 2 a'.c
  int pos[kMaxR];            // last key row r sees (tail-aligned causality); -1 for padding rows
  union {
    float4 xch[2][kTile];    // upper-half partials per token (sum r^2 (K - 2 a'.v), sum r^2, |v - c|^2 part, singular)
    struct {                 // after the last tile (dominant mode): per-lane-quarter sums
      float red[4][kMaxR], red2[4][kMaxR], ltot[kMaxR];
    } fx;
  };
  unsigned long long domf;   // bit r: row r's dominant key lies in this CTA's split (dominant mode)
  int domj[kMaxR];           // position of that key (found while scoring; -1 before)
  float dome[kMaxR];         // its e
  alignas(16) float cf[kDPad];   // the shift c (bf16 values) as f32
  int shift;                 // 1: |v - c|^2 with this c; 0: c = 0 and |v|^2
};

template <int NR, bool SNAP>
constexpr int pass2_smem_bytes() {
  return Pass2Cfg<NR, SNAP>::kOffSmall + (int)sizeof(Pass2Small) + 1024;
}

// Splits pass 1 gave a unit of a sequence of length nb (as its grid share
// computed them).  Warp-collective.
__device__ __forceinline__ int pass1_splits(const AttnParams& p, int nb) {
  if (p.part_splits > 0) return p.part_splits;   // the window states came from elsewhere (prefill)
  if (p.even > 0) return p.even;
  const int tiles = seq_tiles(p, nb);
  const uint32_t tot = total_tiles(p);
  const uint32_t extra = (uint32_t)(p.ctas - p.U);
  const int s = extra ? 1 + (int)(extra * (uint32_t)tiles / tot) : 1;
  return min(min(p.splits1, tiles), s);
}

// acc + (v0^2, v1^2) for the bf16 pair w = (v0, v1) (packed f32x2)
__device__ __forceinline__ uint64_t sq_bf16x2(uint32_t w, uint64_t acc) {
  const uint64_t v = f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return f2_fma(v, v, acc);
}
// acc + ((v0 - c0)^2, (v1 - c1)^2) for the bf16 pair w = (v0, v1) (packed
// f32x2; the differences of bf16 values are exact in fp32)
__device__ __forceinline__ uint64_t sqdiff_bf16x2(uint32_t w, float c0, float c1, uint64_t acc) {
  const uint64_t dv = f2_sub(f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)), f2_pack(c0, c1));
  return f2_fma(dv, dv, acc);
}

#ifdef DROPKV_TEST_HOOKS
// Test build only: the (unit, tile) whose K copy the scoring pass leaves out,
// so that the MMA issuer's bounded wait for it runs out and the pipeline takes
// its timeout exit.  {-1, -1}: none.
__device__ int g_test_skip_k[2] = {-1, -1};
#endif

// TMA producer (one lane): fills the K ring (and the V ring when HAS_V) tile
// by tile; each slot also carries its tile index, -1 ending the stream.
// dynamic: tiles claimed from the unit's counter (the first claim is passed
// in); otherwise the range [t0, t1).  Returns false after a timeout.
template <int KS, bool HAS_V>
__device__ __forceinline__ bool p2_produce(uint8_t* sK, uint8_t* sV, Pass2Small& S, const CUtensorMap* tmk,
                                           const CUtensorMap* tmv, uint32_t* ctr, int unit, int ntiles, int VS,
                                           bool dynamic, int first, int t0, int t1, uint32_t* status) {
  int issued = 0;
  bool ok = true;
  int vs = 0;            // V slot of tile i (VS is set at run time) and the ring's wraps so far
  uint32_t vwrap = 0;
  for (int i = 0;; ++i) {
    const int ks = i % KS;
    if (i >= KS && !mbar_wait(&S.kempty[ks], ((i / KS) + 1) & 1, &S.abort)) { ok = false; break; }
    if (i >= VS && !mbar_wait(&S.vempty[vs], (vwrap + 1) & 1, &S.abort)) { ok = false; break; }
    const int tile = dynamic ? (i == 0 ? first : (int)atomicAdd(ctr, 1u)) : (t0 + i < t1 ? t0 + i : ntiles);
    if (tile >= ntiles) {
      S.ktile[ks] = -1;
      S.vtile[vs] = -1;
      mbar_arrive(&S.kfull[ks]);
      mbar_arrive(&S.vfull[vs]);
      break;
    }
    S.ktile[ks] = tile;
    S.vtile[vs] = tile;
#ifdef DROPKV_TEST_HOOKS
    if (unit != g_test_skip_k[0] || tile != g_test_skip_k[1])   // the test build may leave one K copy out
#endif
    {
      mbar_arrive_expect_tx(&S.kfull[ks], kTileBytes);
      tma_load_3d(sK + ks * kTileBytes, tmk, &S.kfull[ks], 0, tile * kTile, unit);
      tma_load_3d(sK + ks * kTileBytes + kHalfTile, tmk, &S.kfull[ks], 64, tile * kTile, unit);
    }
    if (!HAS_V) {
      mbar_arrive(&S.vfull[vs]);
    } else {
      mbar_arrive_expect_tx(&S.vfull[vs], kTileBytes);
      tma_load_3d(sV + vs * kTileBytes, tmv, &S.vfull[vs], 0, tile * kTile, unit);
      tma_load_3d(sV + vs * kTileBytes + kHalfTile, tmv, &S.vfull[vs], 64, tile * kTile, unit);
    }
    ++issued;
    if (++vs == VS) {
      vs = 0;
      ++vwrap;
    }
  }
  if (!ok) {
    S.abort = 1;
    atomicOr(status, DROPKV_FLAG_TIMEOUT);
    // wait (bounded) for this CTA's copies still in flight
    for (int i = max(0, issued - KS); i < issued; ++i) mbar_drain(&S.kfull[i % KS], (i / KS) & 1);
    if (HAS_V)
      for (int i = max(0, issued - VS); i < issued; ++i) mbar_drain(&S.vfull[i % VS], (i / VS) & 1);
  }
  return ok;
}

// MMA issuer (one lane): S^T = K Q^T into one of two accumulator pairs and
// A.V^T = V a'_hi^T + V a'_lo^T beside it (not for the SnapKV kind); in the
// dominant mode also O_rest^T += V^T P^T, one tile behind (the workers write
// P from the tile's S).  A V stage is released after its last MMA.  Returns
// false after a timeout.
template <int NR, int KS, bool SNAP>
__device__ __forceinline__ bool p2_mma(const uint8_t* sK, const uint8_t* sV, const uint8_t* sP, Pass2Small& S,
                                       uint32_t tmem, uint32_t qaddr, uint32_t ahi, uint32_t alo, int VS, bool dom) {
  const uint32_t idS = umma_idesc_bf16(128, NR, 0, 0);
  const uint32_t idO = umma_idesc_bf16(128, NR, 1, 1);
  const uint32_t tO = tmem + 4 * NR;
  // O_rest^T += V_t^T P_t^T for tile t held in V slot `slot`
  auto pv = [&](int t, int slot) -> bool {
    if (!mbar_wait(&S.pfull, t & 1, &S.abort)) return false;
    tc_fence_after();
    const uint32_t vb = smem_addr(sV + slot * kTileBytes);
    const uint32_t phi = smem_addr(sP), plo = smem_addr(sP + kTile * NR * 2);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      umma_bf16(tO, desc_mnmajor_sw128(vb, kTile, s), desc_mnmajor_interleave(phi, NR, s), idO, (t > 0 || s > 0));
#pragma unroll
    for (int s = 0; s < 8; ++s)
      umma_bf16(tO, desc_mnmajor_sw128(vb, kTile, s), desc_mnmajor_interleave(plo, NR, s), idO, 1);
    umma_commit(&S.pempty);
    umma_commit(&S.vempty[slot]);
    return true;
  };
  int vs = 0, pvs = 0;     // V slots of tiles i and i - 1 (VS is set at run time)
  uint32_t vwrap = 0;
  int i = 0;
  for (;; ++i) {
    const int ks = i % KS, ab = i & 1;
    const uint32_t dS = tmem + ab * 2 * NR, dAV = dS + NR;
    if (!mbar_wait(&S.kfull[ks], (i / KS) & 1, &S.abort)) return false;
    if (*reinterpret_cast<volatile int*>(&S.ktile[ks]) < 0) break;     // no more tiles
    if (i >= 2 && !mbar_wait(&S.accempty[ab], ((i >> 1) + 1) & 1, &S.abort)) return false;
    tc_fence_after();
    const uint32_t kb = smem_addr(sK + ks * kTileBytes);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      umma_bf16(dS, desc_kmajor_sw128(kb, kTile, s), desc_kmajor_sw128(qaddr, NR, s), idS, s > 0);
    umma_commit(&S.kempty[ks]);
    if (SNAP) {
      umma_commit(&S.accfull[ab]);
      continue;
    }
    if (i == 0 && !mbar_wait(&S.aready, 0, &S.abort)) return false;
    if (!mbar_wait(&S.vfull[vs], vwrap & 1, &S.abort)) return false;
    tc_fence_after();
    const uint32_t vb = smem_addr(sV + vs * kTileBytes);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      umma_bf16(dAV, desc_kmajor_sw128(vb, kTile, s), desc_kmajor_sw128(ahi, NR, s), idS, s > 0);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      umma_bf16(dAV, desc_kmajor_sw128(vb, kTile, s), desc_kmajor_sw128(alo, NR, s), idS, 1);
    if (!dom) umma_commit(&S.vempty[vs]);
    umma_commit(&S.accfull[ab]);
    if (dom && i > 0 && !pv(i - 1, pvs)) return false;
    pvs = vs;
    if (++vs == VS) {
      vs = 0;
      ++vwrap;
    }
  }
  if (dom && i > 0 && !pv(i - 1, pvs)) return false;
  return true;
}

// Worker prologue (after the merge): the merged a' = a - c (bf16 hi + lo,
// the A.V^T operand), the per-row constants, the head's shift c and the
// dominated rows whose key lies in this CTA's split.
template <int NR, bool SNAP>
__device__ __forceinline__ void p2_prologue(uint8_t* sAhi, uint8_t* sAlo, Pass2Small& S, const AttnParams& p, int unit, int split,
                            int nb, int tid) {
  const int R = p.R;
  const size_t rowbase = (size_t)unit * R;
  if (!SNAP) {
    const __nv_bfloat16* ahl = p.ahl + (size_t)unit * 2 * kMaxR * kDPad;
    stage_rows_sw128(sAhi, ahl, NR, NR, kDPad, kDPad, tid, kWorkers);
    stage_rows_sw128(sAlo, ahl + kMaxR * kDPad, NR, NR, kDPad, kDPad, tid, kWorkers);
    if (tid < kDPad) S.cf[tid] = p.cvec[(size_t)unit * kDPad + tid];
    if (tid == 0) S.shift = p.cflag[unit];
    fence_proxy_async_smem();
  }
  if (tid < kMaxR) {
    const bool real = tid < R;
    const size_t o = rowbase + tid;
    float* pm = reinterpret_cast<float*>(&S.pml[tid >> 1]);
    pm[tid & 1] = real ? -p.m2[o] : 0.f;
    pm[2 + (tid & 1)] = real ? p.l[o] : 1.f;
    reinterpret_cast<float*>(&S.pk[tid >> 1])[tid & 1] = (!SNAP && real) ? p.aa[o] : 0.f;
    S.pos[tid] = real ? nb - p.w + (tid % p.w) : -1;
    const bool mine = !SNAP && real && p.dom_s[o] == split;
    const unsigned ballot_lo = __ballot_sync(0xffffffffu, mine);   // tid < 64: warps 0 and 1, whole warps
    if (tid == 0) reinterpret_cast<unsigned*>(&S.domf)[0] = ballot_lo;
    if (tid == 32) reinterpret_cast<unsigned*>(&S.domf)[1] = ballot_lo;
    S.domj[tid] = -1;
  }
}

// Score workers: thread (quarter wq, half) owns token wq*32 + lane of each
// tile, rows [r0, r0 + HR) and columns [64 half, 64 half + 64) of |v - c|^2;
// the upper half hands its partial sums to the lower half, which writes the
// score.  DOM: the dominant mode (P for O_rest, the dominant keys' terms at the
// end).  SHIFT: 0 |v|^2 (the head is not shifted), 1 |v - c|^2, 2 either, as
// the head says (the dominant mode); a CTA's hot loop holds one variant only.
// Returns true when a wait gave up.
template <int NR, int VS, bool SNAP, bool DOM, int SHIFT>
__device__ __forceinline__ bool p2_work(uint8_t* sV, uint8_t* sP, Pass2Small& S, const AttnParams& p, uint32_t tmem, int unit,
                        int nb, int tid, uint32_t& flags) {
  constexpr int HR = NR / 2;
  constexpr int kPBytes = kTile * NR * 2;
  const int warp = tid >> 5, lane = tid & 31;
  const int wq = warp & 3, half = warp >> 2;
  const int tok = wq * 32 + lane;
  const int r0 = half * HR;
  const int R = p.R;
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  uint32_t rowmask = 0, dommask = 0;
#pragma unroll
  for (int r = 0; r < HR; ++r) rowmask |= (uint32_t)(r0 + r < R) << r;
  if (DOM) {
#pragma unroll
    for (int r = 0; r < HR; ++r) dommask |= (uint32_t)((S.domf >> (r0 + r)) & 1ull) << r;
  }
  float lrest[DOM ? HR : 1];
#pragma unroll
  for (int r = 0; r < (DOM ? HR : 1); ++r) lrest[r] = 0.f;
  const float scale = p.scale_log2;
  const float inv_g = 1.0f / (float)p.g;
  const int all_see = nb - p.w;
  const bool shifted = SHIFT == 1 || (SHIFT == 2 && S.shift != 0);
  float* raw = p.raw + (size_t)unit * p.n_max;
  bool failed = false;
  for (int i = 0;; ++i) {
    const int vs = i % VS, ab = i & 1;
    // the V slot carries the tile index (and, in the SnapKV mode, nothing else)
    bool ok = __all_sync(0xffffffffu, mbar_wait(&S.vfull[vs], (i / VS) & 1, &S.abort));
    const int tile = ok ? *reinterpret_cast<volatile int*>(&S.vtile[vs]) : 0;
    const bool stop = ok && tile < 0;             // no more tiles (the same slot for every worker)
    const int tile0 = max(tile, 0) * kTile;
    const int j = tile0 + tok;
    const bool full = tile0 + kTile - 1 <= all_see;
    uint8_t* vrow = sV + vs * kTileBytes + half * kHalfTile + tok * 128;
    float vvh = 0.f;
    if (!SNAP && ok && !stop) {
      // |v - c|^2 (or |v|^2 when the head is not shifted) over this half's 64
      // columns, two columns per packed instruction; the chunks are visited in
      // a per-thread rotated order so a warp's reads spread over all banks
      // (physical chunk pc of swizzled row tok holds columns 8 (pc ^ (tok & 7)) .. + 7)
      uint64_t acc = 0, accb = 0;    // two accumulators: shorter dependency chains
      if (SHIFT != 0 && (SHIFT == 1 || shifted)) {
        const float* cfh = S.cf + half * 64;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int pc = (c + tok) & 7, lc = pc ^ (tok & 7);
          const uint4 w = *reinterpret_cast<const uint4*>(vrow + pc * 16);
          const float4 c0 = *reinterpret_cast<const float4*>(cfh + lc * 8);
          const float4 c1 = *reinterpret_cast<const float4*>(cfh + lc * 8 + 4);
          acc = sqdiff_bf16x2(w.x, c0.x, c0.y, acc);
          accb = sqdiff_bf16x2(w.y, c0.z, c0.w, accb);
          acc = sqdiff_bf16x2(w.z, c1.x, c1.y, acc);
          accb = sqdiff_bf16x2(w.w, c1.z, c1.w, accb);
        }
      } else if (SHIFT != 1) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w = *reinterpret_cast<const uint4*>(vrow + ((c + tok) & 7) * 16);
          acc = sq_bf16x2(w.x, acc);
          accb = sq_bf16x2(w.y, accb);
          acc = sq_bf16x2(w.z, acc);
          accb = sq_bf16x2(w.w, accb);
        }
      }
      acc = f2_add(acc, accb);
      vvh = f2_lo(acc) + f2_hi(acc);
    }
    __syncwarp();
    if (lane == 0 && !stop) mbar_arrive(&S.vempty[vs]);
    if (ok && !stop) ok = mbar_wait(&S.accfull[ab], (i >> 1) & 1, &S.abort);
    ok = __all_sync(0xffffffffu, ok);
    // dominant mode: the P buffer is free once the previous tile's PV is done
    if (DOM && ok && !stop && i > 0) ok = __all_sync(0xffffffffu, mbar_wait(&S.pempty, (i - 1) & 1, &S.abort));
    float A = 0.f, W = 0.f;
    bool singular = false;
    if (ok && !stop) {
      tc_fence_after();
      const uint32_t tS = tmem + lane_base + ab * 2 * NR + r0, tAV = tS + NR;
      uint32_t vis = rowmask;
      if (!full) {
        uint32_t v = 0;
        if (j < nb) {
#pragma unroll
          for (int r = 0; r < HR; ++r) v |= (uint32_t)(j <= S.pos[r0 + r]) << r;
        }
        vis &= v;
      }
      if (SNAP) {
        // SnapKV: A accumulates p_j = e / L over the visible rows
        float sv[HR];
        tmem_ld_cols<HR>(tS, sv);
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < HR; ++r)
          if ((vis >> r) & 1u) {
            const float4 c = S.pml[(r0 + r) >> 1];
            A = fmaf(ex2_approx(fmaf(sv[r], scale, (r & 1) ? c.y : c.x)), rcp_approx((r & 1) ? c.w : c.z), A);
          }
      } else if (!DOM) {
        // two rows per packed instruction, in groups of 16 rows (fewer live
        // registers); rows the token is invisible to get e = 0 (their terms
        // vanish; slots past the sequence are never written)
        constexpr int CH = HR < 16 ? HR : 16;
        uint64_t A2 = 0, W2 = 0, A2b = 0, W2b = 0;    // alternate pairs: shorter chains
        const uint64_t scale2 = f2_pack(scale, scale), neg2 = f2_pack(-2.f, -2.f);
#pragma unroll
        for (int c0 = 0; c0 < HR; c0 += CH) {
          float sv[CH], av[CH];
          tmem_ld_cols<CH>(tS + c0, sv);
          tmem_ld_cols<CH>(tAV + c0, av);
          tmem_wait_ld();
#pragma unroll
          for (int rr = 0; rr < CH; rr += 2) {
            const int r = c0 + rr;
            const float4 ml = S.pml[(r0 + r) >> 1];
            const float2 kk = S.pk[(r0 + r) >> 1];
            const uint64_t y = f2_fma(f2_pack(sv[rr], sv[rr + 1]), scale2, f2_pack(ml.x, ml.y));
            const float e0 = ((vis >> r) & 1u) ? ex2_approx(f2_lo(y)) : 0.f;
            const float e1 = ((vis >> (r + 1)) & 1u) ? ex2_approx(f2_hi(y)) : 0.f;
            const uint64_t e2 = f2_pack(e0, e1);
            const uint64_t den = f2_sub(f2_pack(ml.z, ml.w), e2);         // L (1 - p_j)
            const float d0 = f2_lo(den), d1 = f2_hi(den);
            singular |= !(d0 > 0.f) || !(d1 > 0.f);
            const uint64_t ratio = f2_mul(e2, f2_pack(rcp_approx(d0), rcp_approx(d1)));   // p_j / (1 - p_j)
            const uint64_t q = f2_mul(ratio, ratio);
            if ((rr & 2) == 0) {
              A2 = f2_fma(q, f2_fma(f2_pack(av[rr], av[rr + 1]), neg2, f2_pack(kk.x, kk.y)), A2);
              W2 = f2_add(W2, q);
            } else {
              A2b = f2_fma(q, f2_fma(f2_pack(av[rr], av[rr + 1]), neg2, f2_pack(kk.x, kk.y)), A2b);
              W2b = f2_add(W2b, q);
            }
          }
        }
        A2 = f2_add(A2, A2b);
        W2 = f2_add(W2, W2b);
        A = f2_lo(A2) + f2_hi(A2);
        W = f2_lo(W2) + f2_hi(W2);
      } else {
        // dominant mode, in groups of 16 rows like the packed path
        constexpr int CH = HR < 16 ? HR : 16;
#pragma unroll
        for (int c0 = 0; c0 < HR; c0 += CH) {
        float sv[CH], av[CH];
        tmem_ld_cols<CH>(tS + c0, sv);
        tmem_ld_cols<CH>(tAV + c0, av);
        tmem_wait_ld();
#pragma unroll
        for (int c8 = c0 / 8; c8 < (c0 + CH) / 8; ++c8) {
          uint32_t hp[4], lp[4];
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) {
            float pe[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int r = c8 * 8 + 2 * q2 + h2;
              const bool vr = (vis >> r) & 1u;
              const float4 ml = S.pml[(r0 + r) >> 1];
              const float2 kk = S.pk[(r0 + r) >> 1];
              const float negm = h2 ? ml.y : ml.x, L = h2 ? ml.w : ml.z, K = h2 ? kk.y : kk.x;
              const float e = vr ? ex2_approx(fmaf(sv[r - c0], scale, negm)) : 0.f;
              // the dominant key of a row this CTA answers for (p > 1/2: unique)
              const bool dp = DOM && vr && ((dommask >> r) & 1u) && e > 0.5f * L;
              if (DOM && dp) {
                S.domj[r0 + r] = j;
                S.dome[r0 + r] = e;
              }
              pe[h2] = dp ? 0.f : e;
              if (DOM) lrest[r] += pe[h2];
              if (vr && !dp) {
                const float den = L - e;                   // L (1 - p_j)
                singular |= !(den > 0.f);
                const float ratio = e * rcp_approx(den);   // p_j / (1 - p_j)
                const float q = ratio * ratio;
                A = fmaf(q, fmaf(-2.f, av[r - c0], K), A);
                W += q;
              }
            }
            if (DOM) split_hi_lo(pe[0], pe[1], hp[q2], lp[q2]);
          }
          if (DOM) {
            const uint32_t off = interleave_mn_offset(tok, r0 + c8 * 8, NR);
            *reinterpret_cast<uint4*>(sP + off) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
            *reinterpret_cast<uint4*>(sP + kPBytes + off) = make_uint4(lp[0], lp[1], lp[2], lp[3]);
          }
        }
        }
        if (DOM && j >= nb) {
          // slots past the sequence may hold anything (NaN): zero this half of
          // their V rows so that 0 * NaN never reaches the O_rest accumulator
          // (the tile's A.V^T has completed and this thread's |v - c|^2 is done)
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      tc_fence_before();
    }
    if (DOM && ok && !stop) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pfull);
    }
    __syncwarp();
    if (lane == 0 && !stop) mbar_arrive(&S.accempty[ab]);
    if (half == 1) S.xch[ab][tok] = make_float4(A, W, vvh, singular ? 1.f : 0.f);
    // one barrier per tile: it carries both "some wait failed" and "no more tiles"
    if (named_bar_or(kBarWork, kWorkers, !ok || stop)) {
      if (named_bar_or(kBarAux, kWorkers, !ok)) failed = true;
      break;
    }
    if (SNAP && half == 0 && j < nb) {
      float s = (A + S.xch[ab][tok].x) * inv_g;
      if (!isfinite(s)) flags |= DROPKV_FLAG_NONFINITE | DROPKV_FLAG_NONFINITE_SCORE;
      raw[j] = s;
    } else if (!SNAP && half == 0 && j < nb) {
      const float4 o = S.xch[ab][tok];
      float s = fmaf(vvh + o.z, W + o.y, A + o.x);
      if (singular || o.w != 0.f) {
        s = INFINITY;
        flags |= DROPKV_FLAG_SINGULAR;
      } else if (!isfinite(s)) {
        flags |= DROPKV_FLAG_NONFINITE | DROPKV_FLAG_NONFINITE_SCORE;
      } else {
        s = fmaxf(s, 0.f) * inv_g;   // the exact value is >= 0; rounding may not make it negative
      }
      raw[j] = s;
    }
  }
  if constexpr (DOM) {
    // The dominant keys' terms.  The MMA warp commits `drain` after its last
    // MMA (the final PV): a single-phase wait.  This code runs once per call
    // on one CTA per head, after the kernel's hot code: it is fetched cold, so
    // it is kept short (loops not unrolled where the body is large) and every
    // global load goes out in one round trip.
    bool okw = true;
    if (!failed) okw = __all_sync(0xffffffffu, mbar_wait(&S.drain, 0, &S.abort));
    if (named_bar_or(kBarWork, kWorkers, failed || !okw)) return true;
    tc_fence_after();
    float o[HR];   // O_rest^T: lane = head dimension tok, columns = rows
    tmem_ld_cols<HR>(tmem + 4 * NR + lane_base + r0, o);
    // Copied to shared memory in one round trip (cp.async, no registers): the
    // merge's O and L of the other splits for every dominated row and its
    // dominant key's V row (warp w: rows w, w + 8, ...; lane: 4 columns), into
    // the V ring, idle now that the last MMA is done: [kMaxR][kDPad] f32 O,
    // [kMaxR][kDPad] bf16 V, [kMaxR] f32 L, then [kMaxR][kDPad] f32 for this
    // thread's O_rest and, in place, its squared differences.  Warp 0 also
    // loads the dominant keys' raw scores.
    float* so = reinterpret_cast<float*>(sV);
    __nv_bfloat16* svs = reinterpret_cast<__nv_bfloat16*>(sV + kMaxR * kDPad * 4);
    float* sdl = reinterpret_cast<float*>(sV + kMaxR * kDPad * 6);
    float* ssq = reinterpret_cast<float*>(sV + kMaxR * kDPad * 6 + kMaxR * 4);
    const size_t rowbase = (size_t)unit * R;
    const int d4 = p.d >> 2;
#pragma unroll 1
    for (int rr = warp; rr < R; rr += kWorkerWarps) {
      const int jst = S.domj[rr];
      if (((S.domf >> rr) & 1ull) && jst >= 0 && lane < d4) {
        cp_async<16>(so + rr * kDPad + 4 * lane, p.dom_o + (rowbase + rr) * p.d + 4 * lane);
        cp_async<8>(svs + rr * kDPad + 4 * lane, p.v + ((size_t)unit * p.n_max + jst) * p.d + 4 * lane);
        if (lane == 0) cp_async<4>(sdl + rr, p.dom_l + rowbase + rr);
      }
    }
    int key[2] = {-1, -1};
    float cur[2] = {0.f, 0.f};
    if (tid < 32) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int rr = lane + 32 * h2;
        key[h2] = (rr < R && ((S.domf >> rr) & 1ull)) ? S.domj[rr] : -1;
        if (key[h2] >= 0) cur[h2] = raw[key[h2]];
      }
    }
    tmem_wait_ld();
    tc_fence_before();
#pragma unroll
    for (int r = 0; r < HR; ++r) {
      const float v = warp_sum(lrest[r]);
      if (lane == 0) S.fx.red[wq][r0 + r] = v;
    }
#pragma unroll
    for (int r = 0; r < HR; ++r) ssq[(r0 + r) * kDPad + tok] = o[r];
    cp_async_wait_all();
    named_bar(kBarAux, kWorkers);
    // (a) every thread: the squared differences of its token for the
    // dominated rows of its half (rows it does not answer for are skipped the
    // same way by the whole warp)
#pragma unroll 1
    for (int r = 0; r < HR; ++r) {
      const int rr = r0 + r;
      if (!((dommask >> r) & 1u) || S.domj[rr] < 0) continue;
      const float lt = sdl[rr] + ((S.fx.red[0][rr] + S.fx.red[1][rr]) + (S.fx.red[2][rr] + S.fx.red[3][rr]));
      float sq = 0.f;
      if (tok < p.d) {
        const float ar = (so[rr * kDPad + tok] + ssq[rr * kDPad + tok]) / lt;
        const float df = ar - __bfloat162float(svs[rr * kDPad + tok]);
        sq = df * df;
      }
      ssq[rr * kDPad + tok] = sq;
      if (tok == 0) S.fx.ltot[rr] = lt;
    }
    named_bar(kBarAux, kWorkers);
    // (b) |a_rest - v*|^2 of each dominated row: 8 threads per row, 16
    // tokens each in order, then a fixed butterfly over the 8
#pragma unroll 1
    for (int rr = tid >> 3; rr < kMaxR; rr += kWorkers / 8) {
      const int part = tid & 7;
      const bool act = rr < R && ((S.domf >> rr) & 1ull) && S.domj[rr] >= 0;
      float sum = 0.f;
      if (act)
        for (int c = part * 16; c < part * 16 + 16 && c < p.d; ++c) sum += ssq[rr * kDPad + c];
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      sum += __shfl_xor_sync(0xffffffffu, sum, 4);
      if (act && part == 0) S.fx.red2[0][rr] = sum;
    }
    named_bar(kBarAux, kWorkers);
    if (tid < 32) {
      // (c) one lane per row (two passes for rows 32 .. 63): the row's term;
      // the terms of the rows that share a dominant key are summed in row
      // order by the first of them, which adds them to the key's score with
      // one write (several rows may share a key)
      float term[2];
      bool sing[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int rr = lane + 32 * h2;
        term[h2] = 0.f;
        sing[h2] = false;
        if (key[h2] >= 0) {
          const float es = S.dome[rr], lt = S.fx.ltot[rr];
          if (!(lt > es * 0x1p-53f)) {   // p* = e* / (e* + L_rest) rounds to 1 in double precision
            sing[h2] = true;
          } else {
            const float pr = es / (es + lt);
            term[h2] = pr * pr * S.fx.red2[0][rr];
          }
        }
      }
#pragma unroll 1
      for (int h2 = 0; h2 < 2 && 32 * h2 < R; ++h2) {
        const int kk = h2 ? key[1] : key[0];
        const int rr = lane + 32 * h2;
        float add = 0.f;
        bool sg = false, first = kk >= 0;
        // rows in order: q < rr with the same key makes this row not the first
#pragma unroll 1
        for (int q = 0; q < R; ++q) {
          const int qh = q >> 5, ql = q & 31;
          const int kq = __shfl_sync(0xffffffffu, qh ? key[1] : key[0], ql);
          const float tq = __shfl_sync(0xffffffffu, qh ? term[1] : term[0], ql);
          const bool sq2 = __shfl_sync(0xffffffffu, (int)(qh ? sing[1] : sing[0]), ql) != 0;
          if (kk >= 0 && kq == kk) {
            if (q < rr) first = false;
            add += tq;
            sg |= sq2;
          }
        }
        if (first) {
          const float c0 = h2 ? cur[1] : cur[0];
          if (sg) {
            raw[kk] = INFINITY;
            flags |= DROPKV_FLAG_SINGULAR;
          } else {
            const float nv = c0 + add * inv_g;
            if (!isfinite(nv) && !isinf(c0)) flags |= DROPKV_FLAG_NONFINITE | DROPKV_FLAG_NONFINITE_SCORE;
            raw[kk] = nv;
          }
        }
      }
    }
  }
  return failed;
}

// The workers of a CTA in the dominant mode, as a function of their own: the
// kernel's main body keeps only the common path's code, next to the prologue
// (instruction fetch of a cold kernel is on pass 2's critical path).
template <int NR>
__device__ __noinline__ bool p2_work_dominant(uint8_t* sV, uint8_t* sP, Pass2Small* S, const AttnParams* p,
                                              uint32_t tmem, int unit, int nb, int tid, uint32_t* flags) {
  return p2_work<NR, Pass2Dom<NR>::VS, false, true, 2>(sV, sP, *S, *p, tmem, unit, nb, tid, *flags);
}
// The same for a head whose scores use the shift (|v - c|^2).
template <int NR>
__device__ __noinline__ bool p2_work_shifted(uint8_t* sV, Pass2Small* S, const AttnParams* p, uint32_t tmem,
                                             int unit, int nb, int tid, uint32_t* flags) {
  return p2_work<NR, Pass2Cfg<NR, false>::VS, false, false, 1>(sV, nullptr, *S, *p, tmem, unit, nb, tid, *flags);
}

// SNAP: the SnapKV score (1/g) sum_r p_r from K alone -- no V, no A V^T.
template <int NR, bool SNAP>
__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                 const AttnParams p) {
  using C = Pass2Cfg<NR, SNAP>;
  using D = Pass2Dom<NR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sQ = sm + C::kOffQ;
  uint8_t* sAhi = sm + C::kOffAhi;
  uint8_t* sAlo = sm + C::kOffAlo;
  Pass2Small& S = *reinterpret_cast<Pass2Small*>(sm + C::kOffSmall);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const CtaWork wk = cta_work(p, blockIdx.x);
  if (wk.unit < 0) return;                   // left over: no work in this pass
  const int unit = wk.unit, nb = wk.nb;
  const int b = unit / p.Hkv, h = unit - b * p.Hkv;
  if (nb < p.w || nb > p.n_max) return;      // flagged by pass 1
  const int R = p.R;
  const int ntiles = ceil_div(nb, kTile);

  if (tid == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&S.kfull[i], 1);
      mbar_init(&S.kempty[i], 1);
      mbar_init(&S.vfull[i], 1);
      mbar_init(&S.vempty[i], kWorkerWarps + (SNAP ? 0 : 1));
    }
    for (int i = 0; i < 2; ++i) { mbar_init(&S.accfull[i], 1); mbar_init(&S.accempty[i], kWorkerWarps); }
    mbar_init(&S.drain, 1);
    mbar_init(&S.aready, 1);
    mbar_init(&S.pfull, kWorkerWarps);
    mbar_init(&S.pempty, 1);
    S.abort = 0;
    S.mode = kModeDynamic;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&S.tmem_base, C::kTmemCols);
  if (tid < kWorkers) {
    const __nv_bfloat16* qsrc = p.q + ((size_t)b * p.Hq + (size_t)h * p.g) * p.w * p.d;
    stage_rows_sw128(sQ, qsrc, NR, R, p.d, p.d, tid, kWorkers);
    fence_proxy_async_smem();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmk);
    if (!SNAP) tma_prefetch_desc(&tmv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  bool failed = false;
  // The merged statistics of pass 1 are staged by the workers after
  // grid_dep_wait() and released to the MMA warp through `aready`.  The
  // producer also waits: streaming K and V while the merge runs would only
  // slow the merge's loads, on which every worker waits.
  grid_dep_launch();

  if (warp == kProducerWarp) {
    grid_dep_wait();                              // the merge's outputs and the cleared tile counter
    int mode = kModeDynamic, first = 0, t0 = 0, t1 = 0;
    if (lane == 0) first = (int)atomicAdd(p.tile_ctr + unit, 1u);   // in flight with the loads below
    if constexpr (!SNAP) {
      const int* ds = p.dom_s + (size_t)unit * R;
      const int s0 = lane < R ? ds[lane] : -1;
      const int s1 = lane + 32 < R ? ds[lane + 32] : -1;
      if (__any_sync(0xffffffffu, s0 >= 0 || s1 >= 0)) {
        const int ns1 = pass1_splits(p, nb);
        mode = __any_sync(0xffffffffu, s0 == wk.split || s1 == wk.split) ? kModeDominant : kModeStatic;
        if (wk.split < ns1) {
          t0 = (int)((uint32_t)wk.split * (uint32_t)ntiles / (uint32_t)ns1);
          t1 = (int)((uint32_t)(wk.split + 1) * (uint32_t)ntiles / (uint32_t)ns1);
        }
      }
    }
    if (lane == 0) {
      S.mode = mode;                              // published by the first slot's arrival
      p2_produce<C::KS, !SNAP>(sm + C::kOffK, sm + C::kOffV, S, &tmk, &tmv, p.tile_ctr + unit, unit, ntiles,
                               (!SNAP && mode == kModeDominant) ? D::VS : C::VS, mode == kModeDynamic, first, t0, t1,
                               p.status);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t qaddr = smem_addr(sQ), ahi = smem_addr(sAhi), alo = smem_addr(sAlo);
      // the first slot (stage 0 in every layout) brings the mode
      bool ok = mbar_wait(&S.kfull[0], 0, &S.abort);
      if (ok) {
        const int mode = *reinterpret_cast<volatile int*>(&S.mode);
        const bool dom = !SNAP && mode == kModeDominant;
        ok = p2_mma<NR, C::KS, SNAP>(sm + C::kOffK, sm + C::kOffV, sm + D::kOffP, S, tmem, qaddr, ahi, alo,
                                     dom ? D::VS : C::VS, dom);
      }
      if (!ok) {
        failed = true;
        S.abort = 1;
        atomicOr(p.status, DROPKV_FLAG_TIMEOUT);
      }
      umma_commit(&S.drain);
      mbar_drain(&S.drain, 0);
    }
    __syncwarp();
  } else if (warp < kWorkerWarps) {
    uint32_t flags = 0;
    grid_dep_wait();                              // a, m, L and the dominated rows come from the merge
    p2_prologue<NR, SNAP>(sAhi, sAlo, S, p, unit, wk.split, nb, tid);
    named_bar(kBarWork, kWorkers);
    if (tid == 0) mbar_arrive(&S.aready);
    // the first slot (stage 0 in every layout) brings the mode; every worker
    // takes the same branch
    const bool ok0 = mbar_wait(&S.vfull[0], 0, &S.abort);
    if (named_bar_or(kBarAux, kWorkers, !ok0)) {
      failed = true;
    } else {
      const int mode = *reinterpret_cast<volatile int*>(&S.mode);
      if (!SNAP && mode == kModeDominant)
        failed = p2_work_dominant<NR>(sm + C::kOffV, sm + D::kOffP, &S, &p, tmem, unit, nb, tid, &flags);
      else if (!SNAP && S.shift)
        failed = p2_work_shifted<NR>(sm + C::kOffV, &S, &p, tmem, unit, nb, tid, &flags);
      else
        failed = p2_work<NR, C::VS, SNAP, false, 0>(sm + C::kOffV, nullptr, S, p, tmem, unit, nb, tid, flags);
    }
    if (flags) atomicOr(p.status, flags);
  }
  if (failed) S.abort = 1;
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int NR, bool SNAP>
cudaError_t launch_pass1_t(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  constexpr int smem = pass1_smem_bytes<NR, SNAP>();
  static_assert(smem <= 232448, "pass-1 shared memory exceeds the per-CTA limit");
  auto kern = window_attention_kernel<NR, SNAP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(p.ctas), dim3(kThreads), smem, st, tk, tv, p);
}

template <int NR, bool SNAP>
cudaError_t launch_pass2_t(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  constexpr int smem = pass2_smem_bytes<NR, SNAP>();
  static_assert(smem <= 232448, "pass-2 shared memory exceeds the per-CTA limit");
  auto kern = score_kernel<NR, SNAP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(p.ctas), dim3(kThreads), smem, st, tk, tv, p);
}


// ============================================================== prefill attention
// Causal attention of every query row of a prompt ("DropKV: Decoupling ...",
// section 2.1): the kernel a scorer fused into prefill lives in.  Its last w
// rows are step S1's window rows, so pass 1 and its read of K and V drop out
// of the eviction.
//
// A CTA holds two 128-row query tiles of one head, one per softmax group of
// four warps; thread t of a group owns TMEM lane t, the whole of its row, so
// the row maximum needs no exchange between threads.  Per key tile:
//   S = Q K^T on tcgen05 (M = 128 rows, N = 128 keys) into the group's 128
//   TMEM columns;  P = 2^(x - ref) with a lazily moved reference as in pass 1,
//   written back over S as bf16 pairs;  O += P V with P read from tensor
//   memory (V from shared memory, MN-major).
// The group's next S is issued after its P V (the tensor core runs one
// thread's MMAs in issue order, so S does not overwrite P before P V has
// read it), and the MMA warp alternates the groups: one group's P V and next
// S run while the other group's softmax works.  The tiles without window
// rows go in pairs (t - 1, t), so the two key ranges differ by one tile.
// The one or two tiles that hold window rows run alone in group 1 of their
// own CTAs (started first: they are the longest): P in bf16 hi and lo parts
// (two P V per key tile) and the accumulator folded every kPfFold key tiles
// into the idle group's O columns, so their output keeps pass 1's precision;
// their rows also write their state in pass 1's partial layout (one partial
// per row) and their query row, for the merge and pass 2.
constexpr int kPfProducerWarp = 8, kPfMmaWarp = 9, kPfThreads = 32 * 12;   // warps 10, 11 idle
constexpr int kPfOffQ = 0, kPfOffK = 2 * kTileBytes, kPfOffV = 4 * kTileBytes, kPfOffSmall = 6 * kTileBytes;
constexpr uint32_t kPfTmemCols = 512;   // group g: S at [128 g, 128 g + 128), O at [256 + 128 g, ...)
// Every kPfFold key tiles the accumulator O of a window tile is folded into
// O2 with fp32 register adds and restarted, so no tensor-core accumulation
// chain runs over more than kPfFold tiles (at n = 32K one chain of 256 tiles
// left the window output 1.7e-4 off in relative terms; pass 1's splits chain
// about 54).
constexpr int kPfFold = 16;

struct PrefillSmem {
  uint64_t qbar, kfull[2], kempty[2], vfull[2], vempty[2];
  uint64_t sfull[2];   // group g: S(i) and every MMA issued before it complete
  uint64_t pfull[2];   // group g: P(i) written by the group's four warps
  uint64_t odone[2];   // group g: its last P V complete
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr int kPfSmem = kPfOffSmall + (int)sizeof(PrefillSmem) + 1024;
static_assert(kPfSmem <= 232448, "prefill shared memory exceeds the per-CTA limit");

// The softmax group of a prefill CTA (warps 4g .. 4g + 3, one row per
// thread); PRECISE: the window tiles' variant (hi and lo parts of P, the
// accumulator fold, the rows' partial states).  One instance per CTA kind
// keeps each loop's code short.
template <bool PRECISE>
__device__ __forceinline__ void prefill_softmax(const PrefillParams& p, PrefillSmem& S, uint8_t* sm, uint32_t tmem,
                                                int warp, int lane, int b, int hq, int unit, int nb, int t0, int t1) {
  const int h = hq / p.g;
  const int g = warp >> 2, quarter = warp & 3;
  const int tg = g ? t1 : t0;
  const int row = quarter * 32 + lane, pos = tg * kTile + row;
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const uint32_t tS = tmem + lane_base + 128 * g, tOg = tmem + lane_base + 256 + 128 * g;
  const uint32_t tO2 = tmem + lane_base + 256;   // window tiles: the idle group 0's O columns
  const float scale = p.scale_log2;
  float ref = -INFINITY, l = 0.f, emax = 0.f;
  // A wait this warp gave up on sets `bad` and raises the timeout flag and
  // the CTA's abort flag, which ends every other wait of the CTA; the warp
  // stops (no further arrivals).
  bool bad = tg < 0;
  auto give_up = [&]() {
    bad = true;
    if (lane == 0) {
      S.abort = 1;
      atomicOr(p.status, DROPKV_FLAG_TIMEOUT);
    }
  };
  for (int i = 0; !bad && i <= tg; ++i) {
    if (!__all_sync(0xffffffffu, mbar_wait(&S.sfull[g], i & 1, &S.abort))) { give_up(); break; }
    tc_fence_after();
    float x[128];
#pragma unroll
    for (int c = 0; c < 8; ++c) tmem_ld16(tS + 16 * c, x + 16 * c);
    tmem_wait_ld();
    if (i == tg) {   // the diagonal tile: keys past the row or the sequence
#pragma unroll
      for (int u = 0; u < 128; ++u) {
        const int j = i * kTile + u;
        if (!(j <= pos && j < nb)) x[u] = -INFINITY;
      }
    }
    // the row's largest raw logit (the scale is positive: applied in the FMA below)
    float m8[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) m8[u] = x[u];
#pragma unroll
    for (int u = 8; u < 128; ++u) m8[u & 7] = fmaxf(m8[u & 7], x[u]);
    const float mt = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                           fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * scale;
    const bool need = mt > ref + kRescaleLog2;
    float factor = 1.f;
    if (need) {
      factor = (ref == -INFINITY) ? 0.f : ex2_approx(ref - mt);
      ref = mt;
      l *= factor;
      emax *= factor;
    }
    // e = 2^(x scale - ref), the exponent two columns per packed FMA, and
    // the row sum over four packed accumulators
    const uint64_t sc2 = f2_pack(scale, scale), nr2 = f2_pack(-ref, -ref);
#pragma unroll
    for (int u = 0; u < 128; u += 2) {
      const uint64_t y = f2_fma(f2_pack(x[u], x[u + 1]), sc2, nr2);
      x[u] = ex2_approx(f2_lo(y));
      x[u + 1] = ex2_approx(f2_hi(y));
    }
    uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int u = 0; u < 128; u += 2) ls2[(u >> 1) & 3] = f2_add(ls2[(u >> 1) & 3], f2_pack(x[u], x[u + 1]));
    const uint64_t lsum = f2_add(f2_add(ls2[0], ls2[1]), f2_add(ls2[2], ls2[3]));
    l += f2_lo(lsum) + f2_hi(lsum);
    if (PRECISE) {   // the largest e is only wanted for window rows
#pragma unroll
      for (int u = 0; u < 128; ++u) emax = fmaxf(emax, x[u]);
    }
    // P over S's columns (all read by now): bf16 pairs at [0, 64), and in
    // window tiles the rounding remainders at [64, 128)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float hw[16], lw[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        uint32_t hi, lo;
        if (PRECISE) {
          split_hi_lo(x[32 * c + 2 * q], x[32 * c + 2 * q + 1], hi, lo);
        } else {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[32 * c + 2 * q], x[32 * c + 2 * q + 1]);
          hi = *reinterpret_cast<const uint32_t*>(&h2);
          lo = 0u;
        }
        hw[q] = __uint_as_float(hi);
        lw[q] = __uint_as_float(lo);
      }
      tmem_st16(tS + 16 * c, hw);
      if (PRECISE) tmem_st16(tS + 64 + 16 * c, lw);
    }
    if (PRECISE && i == 0) {
      // O2 starts at zero (TMEM holds anything after allocation)
      float z[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) z[u] = 0.f;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) tmem_st16(tO2 + 16 * c, z);
    }
    // (after the P stores, so that x is dead) P V(i - 1) is complete (the
    // commit S(i) signalled came after it): at a fold O2 = (O2 + O) * factor and P V(i) restarts O; else O *= factor
    // (and O2 *= factor in window tiles)
    const bool fold = PRECISE && i > 0 && i % kPfFold == 0;   // the same in every thread
    if (fold || (i > 0 && __any_sync(0xffffffffu, need))) {
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float o[16], o2[16];
        tmem_ld16(tOg + 16 * c, o);
        if (PRECISE) tmem_ld16(tO2 + 16 * c, o2);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          o2[u] = (fold ? o2[u] + o[u] : o2[u]) * factor;
          o[u] *= factor;
        }
        if (!fold) tmem_st16(tOg + 16 * c, o);
        if (PRECISE) tmem_st16(tO2 + 16 * c, o2);
      }
    }
    if (PRECISE && (i + 1) * kTile > nb) {
      // the last key tile of a sequence whose length is not a multiple of
      // the tile: slots past it may hold anything (NaN); zero their V rows
      // so that 0 * NaN never reaches the accumulator (uniform over the CTA)
      if (!__all_sync(0xffffffffu, mbar_wait(&S.vfull[i & 1], (i >> 1) & 1, &S.abort))) { give_up(); break; }
      if (i * kTile + row >= nb) {
        uint8_t* vrow = sm + kPfOffV + (i & 1) * kTileBytes + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vrow + kHalfTile + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.pfull[g]);
  }
  // ---------------------------------------------------- epilogue
  if (tg >= 0) {
    const bool okw = !bad && __all_sync(0xffffffffu, mbar_wait(&S.odone[g], 0, &S.abort));
    if (!bad && !okw) give_up();
    if (okw) {
      tc_fence_after();
      const bool row_ok = pos < nb;
      const bool win = PRECISE && row_ok && pos >= nb - p.w;
      const int tw = pos - (nb - p.w);
      const int r = (hq - h * p.g) * p.w + tw;
      const size_t part = (size_t)unit * p.splits;          // the single partial of the row
      const float inv_l = 1.0f / l;
      __nv_bfloat16* orow = p.out + (((size_t)b * p.Hq + hq) * p.n_max + pos) * p.d;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float o[16], o2[16];
        tmem_ld16(tOg + 16 * c, o);
        if (PRECISE) tmem_ld16(tO2 + 16 * c, o2);
        tmem_wait_ld();
        if (PRECISE) {
#pragma unroll
          for (int u = 0; u < 16; ++u) o[u] += o2[u];
        }
        const int c0 = 16 * c;
        if (row_ok && c0 < p.d) {
          uint32_t w8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * u] * inv_l, o[2 * u + 1] * inv_l);
            w8[u] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(orow + c0) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
          if (c0 + 8 < p.d) *reinterpret_cast<uint4*>(orow + c0 + 8) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
          if (win) {
            float* po = p.part_o + (part * p.R + r) * p.d + c0;
#pragma unroll
            for (int u = 0; u < 16; u += 4)
              if (c0 + u < p.d) *reinterpret_cast<float4*>(po + u) = make_float4(o[u], o[u + 1], o[u + 2], o[u + 3]);
          }
        }
      }
      if (win) {
        reinterpret_cast<float4*>(p.part_ml)[part * p.R + r] = make_float4(ref, l, emax, 0.f);
        const uint4* qs = reinterpret_cast<const uint4*>(p.q + (((size_t)b * p.Hq + hq) * p.n_max + pos) * p.d);
        uint4* qd = reinterpret_cast<uint4*>(p.q_win + (((size_t)b * p.Hq + hq) * p.w + tw) * p.d);
        for (int c = 0; c < p.d / 8; ++c) qd[c] = qs[c];
      }
    }
  }
}

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_attention_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  PrefillSmem& S = *reinterpret_cast<PrefillSmem*>(sm + kPfOffSmall);
  grid_dep_wait();                          // the inputs may come from the kernel before
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z, hq = blockIdx.y;
  const int nb = p.lengths ? p.lengths[b] : p.n_max;
  if (nb < p.w || nb > p.n_max) {
    if (tid == 0 && blockIdx.x == 0 && hq == 0) atomicOr(p.status, DROPKV_FLAG_BAD_LENGTH);
    return;
  }
  // Query tiles 0 .. F - 1 hold no window row.  Blocks 0 and 1 take tiles F
  // and F + 1 (those before the sequence's end), blocks 2, 3, ... the pairs
  // (F - 2, F - 1), (F - 4, F - 3), ... down to tile 0.  Group 1 takes t1,
  // group 0 t0 (-1: none).
  const int F = (nb - p.w) / kTile;
  const bool precise = blockIdx.x < 2;
  const int t1 = precise ? F + (int)blockIdx.x : F - 1 - 2 * ((int)blockIdx.x - 2);
  const int t0 = precise ? -1 : t1 - 1;
  if (t1 < 0 || t1 * kTile >= nb) return;
  const int h = hq / p.g, unit = b * p.Hkv + h;
  const int nk = t1 + 1;                    // key tiles 0 .. t1 (causal)

  if (tid == 0) {
    mbar_init(&S.qbar, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.kfull[i], 1); mbar_init(&S.kempty[i], 1);
      mbar_init(&S.vfull[i], 1); mbar_init(&S.vempty[i], 1);
      mbar_init(&S.sfull[i], 1); mbar_init(&S.pfull[i], 4);
      mbar_init(&S.odone[i], 1);
    }
    mbar_init(&S.drain, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == kPfMmaWarp) tmem_alloc(&S.tmem_base, kPfTmemCols);
  if (warp == kPfProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  grid_dep_launch();

  if (warp == kPfProducerWarp) {
    if (lane == 0) {
      const int zq = b * p.Hq + hq;
      mbar_arrive_expect_tx(&S.qbar, (t0 >= 0 ? 2 : 1) * kTileBytes);
      if (t0 >= 0) {
        tma_load_3d(sm + kPfOffQ, &tmq, &S.qbar, 0, t0 * kTile, zq);
        tma_load_3d(sm + kPfOffQ + kHalfTile, &tmq, &S.qbar, 64, t0 * kTile, zq);
      }
      tma_load_3d(sm + kPfOffQ + kTileBytes, &tmq, &S.qbar, 0, t1 * kTile, zq);
      tma_load_3d(sm + kPfOffQ + kTileBytes + kHalfTile, &tmq, &S.qbar, 64, t1 * kTile, zq);
      stream_ring<2, true>(sm + kPfOffK, S.kfull, S.kempty, &tmk, 0, nk, unit, 0, &S.abort, p.status);
      mbar_drain(&S.qbar, 0);               // the Q copies have landed before the CTA can leave
    } else if (lane == 1) {
      stream_ring<2>(sm + kPfOffV, S.vfull, S.vempty, &tmv, 0, nk, unit, 0, &S.abort, p.status);
    }
    __syncwarp();
  } else if (warp == kPfMmaWarp) {
    if (lane == 0) {
      const uint32_t idS = umma_idesc_bf16(128, 128, 0, 0);
      const uint32_t idO = umma_idesc_bf16(128, 128, 0, 1);
      const int pps = precise ? 2 : 1;      // P V per key tile: the hi and lo parts in window tiles
      auto issue_S = [&](int g, int i) {    // K tile i has landed
        const uint32_t qa = smem_addr(sm + kPfOffQ + g * kTileBytes);
        const uint32_t kb = smem_addr(sm + kPfOffK + (i & 1) * kTileBytes);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_bf16(tmem + 128 * g, desc_kmajor_sw128(qa, kTile, s), desc_kmajor_sw128(kb, kTile, s), idS, s > 0);
        umma_commit(&S.sfull[g]);
      };
      bool ok = mbar_wait(&S.qbar, 0, &S.abort) && mbar_wait(&S.kfull[0], 0, &S.abort);
      if (ok) {
        tc_fence_after();
        if (t0 >= 0) issue_S(0, 0);
        issue_S(1, 0);
        umma_commit(&S.kempty[0]);
      }
      for (int i = 0; ok && i < nk; ++i) {
        const bool more = i + 1 < nk;
        if (!(ok = mbar_wait(&S.vfull[i & 1], (i >> 1) & 1, &S.abort))) break;
        if (more && !(ok = mbar_wait(&S.kfull[(i + 1) & 1], ((i + 1) >> 1) & 1, &S.abort))) break;
        const uint32_t vb = smem_addr(sm + kPfOffV + (i & 1) * kTileBytes);
        for (int g = 0; g < 2; ++g) {
          const int tg = g ? t1 : t0;
          if (i > tg) continue;             // group 0's tile ends one key tile earlier (or is absent)
          if (!(ok = mbar_wait(&S.pfull[g], i & 1, &S.abort))) break;
          tc_fence_after();
          for (int part = 0; part < pps; ++part) {
#pragma unroll
            for (int s = 0; s < 8; ++s)
              umma_bf16_tmem_a(tmem + 256 + 128 * g, tmem + 128 * g + 64 * part + 8 * s,
                               desc_mnmajor_sw128(vb, kTile, s), idO,
                               precise ? (part > 0 || i % kPfFold != 0 || s > 0) : (i > 0 || s > 0));
          }
          if (i < tg) issue_S(g, i + 1);    // overwrites P(i) after P V(i) has read it
          else umma_commit(&S.odone[g]);
        }
        if (!ok) break;
        if (more) umma_commit(&S.kempty[(i + 1) & 1]);
        umma_commit(&S.vempty[i & 1]);
      }
      if (!ok) {
        S.abort = 1;
        atomicOr(p.status, DROPKV_FLAG_TIMEOUT);
      }
      // no MMA may still be writing TMEM when it is released
      umma_commit(&S.drain);
      mbar_drain(&S.drain, 0);
    }
    __syncwarp();
  } else if (warp < 8) {
    if (precise) prefill_softmax<true>(p, S, sm, tmem, warp, lane, b, hq, unit, nb, t0, t1);
    else prefill_softmax<false>(p, S, sm, tmem, warp, lane, b, hq, unit, nb, t0, t1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kPfMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kPfTmemCols);
  }
}
}  // namespace

cudaError_t launch_window_attention(const AttnParams& p, int NR, const CUtensorMap& tk, const CUtensorMap& tv,
                                    int, cudaStream_t st) {
  const bool snap = p.kind == kKindSnapKV;
  switch (NR) {
    case 16: return snap ? launch_pass1_t<16, true>(p, tk, tv, st) : launch_pass1_t<16, false>(p, tk, tv, st);
    case 32: return snap ? launch_pass1_t<32, true>(p, tk, tv, st) : launch_pass1_t<32, false>(p, tk, tv, st);
    case 64: return snap ? launch_pass1_t<64, true>(p, tk, tv, st) : launch_pass1_t<64, false>(p, tk, tv, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_merge(const AttnParams& p, cudaStream_t st) {
  // row groups covering the NR rows of the A.V^T operand (rows past R get
  // zeros); shared memory for the O columns of up to 32 splits per row
  const size_t smem = (p.kind == kKindSnapKV) ? 0 : (size_t)kMergeRows * std::min(32, p.splits) * 32 * sizeof(float4);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(merge_splits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(merge_splits_kernel, dim3(p.NR / kMergeRows, p.U), dim3(kMergeThreads), smem, st, p);
}

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(prefill_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
  if (e != cudaSuccess) return e;
  // two blocks for the tiles holding window rows, then one per pair of the others
  const dim3 grid(2 + (p.n_max / kTile + 1) / 2, p.Hq, p.B);
  return launch_pdl(prefill_attention_kernel, grid, dim3(kPfThreads), kPfSmem, st, tq, tk, tv, p);
}

cudaError_t launch_score(const AttnParams& p, int NR, const CUtensorMap& tk, const CUtensorMap& tv,
                         cudaStream_t st) {
  const bool snap = p.kind == kKindSnapKV;
  switch (NR) {
    case 16: return snap ? launch_pass2_t<16, true>(p, tk, tv, st) : launch_pass2_t<16, false>(p, tk, tv, st);
    case 32: return snap ? launch_pass2_t<32, true>(p, tk, tv, st) : launch_pass2_t<32, false>(p, tk, tv, st);
    case 64: return snap ? launch_pass2_t<64, true>(p, tk, tv, st) : launch_pass2_t<64, false>(p, tk, tv, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dropkv

#ifdef DROPKV_TEST_HOOKS
#include "dropkv_test_hooks.h"
extern "C" dropkv_status dropkv_test_skip_pass2_k(int32_t unit, int32_t tile) {
  const int v[2] = {unit, tile};
  return cudaMemcpyToSymbol(dropkv::g_test_skip_k, v, sizeof v) == cudaSuccess ? DROPKV_OK : DROPKV_ERR_CUDA;
}
extern "C" dropkv_status dropkv_test_skip_prefill_k(int32_t unit, int32_t tile) {
  const int v[2] = {unit, tile};
  return cudaMemcpyToSymbol(dropkv::g_test_skip_pf_k, v, sizeof v) == cudaSuccess ? DROPKV_OK : DROPKV_ERR_CUDA;
}
#endif
