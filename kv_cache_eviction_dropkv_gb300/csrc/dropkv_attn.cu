// Pass 1 (window attention with split-K and a last-CTA merge) and pass 2
// (streaming per-token perturbation score) of the DropKV scoring path.
//
// Both passes stream 128-token K/V tiles of one KV head through TMA into
// 128-byte-swizzled shared memory and put the two small contractions on the
// tcgen05 tensor cores with fp32 accumulators in TMEM:
//   S^T [128 tokens x R rows] = K_tile . Q^T        (A = K, K-major; B = Q, K-major)
//   pass 1: O^T [128 dims x R] += V_tile^T . P^T     (A = V, MN-major; B = P, MN-major)
//   pass 2: AV^T [128 tokens x R] = V_tile . a^T     (A = V, K-major; B = a_hi, then a_lo)
// with one TMEM lane per token (or per head dimension for O), so each of the
// 128 softmax / score threads owns one token and needs no cross-thread
// reduction on the hot path.
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
#include <cuda_runtime.h>

#include "dropkv_internal.cuh"
#include "sm103_ptx.cuh"

namespace dropkv {
namespace {

constexpr int kWorkers = 128;            // warps 0-3: one thread per TMEM lane
constexpr int kThreads = 192;            // + warp 4 (TMA producer) + warp 5 (MMA issuer, TMEM owner)
constexpr int kTileBytes = kTile * kDPad * 2;   // 32 KB: one K or V tile, two SW128 blocks
constexpr int kHalfTile = kTileBytes / 2;
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

// Wait for a TMA copy to land without honouring the abort flag (used only to
// drain copies in flight before the CTA exits).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kDrainNs) break;
  }
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

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// ============================================================== pass 1
template <int NR>
struct Pass1Cfg {
  static constexpr int KS = NR <= 32 ? 3 : 2;       // K ring depth
  static constexpr int VS = 2;                      // V ring depth
  static constexpr int kQBytes = NR * kDPad * 2;
  static constexpr int kPBytes = kTile * NR * 2;    // one of (hi, lo) of one P buffer
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + KS * kTileBytes;
  static constexpr int kOffQ = kOffV + VS * kTileBytes;
  static constexpr int kOffP = kOffQ + kQBytes;     // [buffer 0, 1][hi, lo]
  static constexpr int kOffSmall = kOffP + 4 * kPBytes;
  static constexpr uint32_t kTmemCols = (3 * NR <= 64) ? 64u : (3 * NR <= 128 ? 128u : 256u);
};

struct Pass1Small {
  uint64_t kfull[3], kempty[3], vfull[2], vempty[2];
  uint64_t sfull[2], sempty[2], pfull[2], pempty[2], ofull, drain;
  uint32_t tmem_base;
  int abort;
  int is_last;
  int pos[kMaxR];          // last key visible to row r (tail-aligned causality)
  float mref[kMaxR];       // current exponent reference of row r (log2 units)
  float red[4][kMaxR];     // per-warp reduction scratch
};

template <int NR>
constexpr int pass1_smem_bytes() {
  return Pass1Cfg<NR>::kOffSmall + (int)sizeof(Pass1Small) + 1024;
}

// Merge the split-K partial states of one KV head (executed by the last CTA).
// m = max_s m_s;  L = sum_s l_s 2^(m_s - m);  a = sum_s O_s 2^(m_s - m) / L.
__device__ void merge_unit(const AttnParams& p, int unit, float* wts, float* Ms, float* Ls, int tid) {
  const int S = p.splits, R = p.R, d = p.d;
  const float* ml = p.part_ml + (size_t)unit * S * R * 2;
  const float* po = p.part_o + (size_t)unit * S * R * d;
  if (tid < R) {
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) {
      const float ls = ml[((size_t)s * R + tid) * 2 + 1];
      if (ls > 0.f) M = fmaxf(M, ml[((size_t)s * R + tid) * 2]);
    }
    float L = 0.f;
    for (int s = 0; s < S; ++s) {
      const float ms = ml[((size_t)s * R + tid) * 2], ls = ml[((size_t)s * R + tid) * 2 + 1];
      const float wgt = (ls > 0.f) ? exp2f(ms - M) : 0.f;
      wts[s * R + tid] = wgt;
      L += ls * wgt;
    }
    Ms[tid] = M;
    Ls[tid] = L;
    if (!(L > 0.f) || !isfinite(L)) atomicOr(p.status, DROPKV_FLAG_NONFINITE);
  }
  __syncthreads();
  float* a_out = p.a + (size_t)unit * R * d;
  for (int idx = tid; idx < R * d; idx += kThreads) {
    const int r = idx / d, c = idx - r * d;
    float acc = 0.f;
    for (int s = 0; s < S; ++s) acc += po[((size_t)s * R + r) * d + c] * wts[s * R + r];
    a_out[idx] = acc / Ls[r];
  }
  __syncthreads();
  // |a|^2, the hi/lo bf16 split of a (zero-padded to [NR pad 64][128]), and the stats
  __nv_bfloat16* ahl = p.ahl + (size_t)unit * 2 * kMaxR * kDPad;
  for (int idx = tid; idx < kMaxR * kDPad; idx += kThreads) {
    const int r = idx / kDPad, c = idx - r * kDPad;
    const float x = (r < R && c < d) ? a_out[r * d + c] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
    ahl[idx] = hi;
    ahl[kMaxR * kDPad + idx] = lo;
  }
  if (tid < R) {
    float aa = 0.f;
    for (int c = 0; c < d; ++c) {
      const float x = a_out[tid * d + c];
      aa = fmaf(x, x, aa);
    }
    const size_t o = (size_t)unit * R + tid;
    p.aa[o] = aa;
    p.m2[o] = Ms[tid];
    p.l[o] = Ls[tid];
    // exported: log-sum-exp of the natural-unit logits, log(L) + m ln 2
    p.m[o] = (Ms[tid] + log2f(Ls[tid])) * 0.69314718055994531f;
    if (!isfinite(aa)) atomicOr(p.status, DROPKV_FLAG_NONFINITE);
  }
}

template <int NR>
__global__ void __launch_bounds__(kThreads, 1)
    window_attention_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                            const AttnParams p) {
  using C = Pass1Cfg<NR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sK = sm + C::kOffK;
  uint8_t* sV = sm + C::kOffV;
  uint8_t* sQ = sm + C::kOffQ;
  uint8_t* sP = sm + C::kOffP;
  Pass1Small& S = *reinterpret_cast<Pass1Small*>(sm + C::kOffSmall);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, unit = blockIdx.y;
  const int b = unit / p.Hkv, h = unit - b * p.Hkv;
  const int nb = p.lengths ? p.lengths[b] : p.n_max;
  if (nb < p.w || nb > p.n_max) {           // invalid length: the unit is skipped
    if (tid == 0 && split == 0 && h == 0) atomicOr(p.status, DROPKV_FLAG_BAD_LENGTH);
    return;
  }
  const int R = p.R;
  const int t0 = split * p.tpc;
  const int t1 = min(t0 + p.tpc, ceil_div(nb, kTile));
  const int T = max(0, t1 - t0);

  if (tid == 0) {
    for (int i = 0; i < C::KS; ++i) { mbar_init(&S.kfull[i], 1); mbar_init(&S.kempty[i], 1); }
    for (int i = 0; i < C::VS; ++i) { mbar_init(&S.vfull[i], 1); mbar_init(&S.vempty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.sfull[i], 1); mbar_init(&S.sempty[i], 4);
      mbar_init(&S.pfull[i], 4); mbar_init(&S.pempty[i], 1);
    }
    mbar_init(&S.ofull, 1);
    mbar_init(&S.drain, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (tid < kMaxR) {
    S.pos[tid] = (tid < R) ? nb - p.w + (tid % p.w) : -1;
    S.mref[tid] = -INFINITY;
  }
  if (T > 0) {
    if (warp == 5) tmem_alloc(&S.tmem_base, C::kTmemCols);
    if (tid < kWorkers) {
      const __nv_bfloat16* qsrc = p.q + ((size_t)b * p.Hq + (size_t)h * p.g) * p.w * p.d;
      stage_rows_sw128(sQ, qsrc, NR, R, p.d, p.d, tid, kWorkers);
      fence_proxy_async_smem();
    }
    if (warp == 4 && lane == 0) { tma_prefetch_desc(&tmk); tma_prefetch_desc(&tmv); }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const uint32_t tS = tmem, tO = tmem + 2 * NR;    // S buffers at [0, 2NR), O at [2NR, 3NR)
  bool failed = false;

  if (T > 0 && warp == 4) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      int issued_k = 0, issued_v = 0;
      for (int i = 0; i < T; ++i) {
        const int y = (t0 + i) * kTile;
        const int ks = i % C::KS, vs = i % C::VS;
        if (i >= C::KS && !mbar_wait(&S.kempty[ks], ((i / C::KS) + 1) & 1, &S.abort)) { failed = true; break; }
        mbar_arrive_expect_tx(&S.kfull[ks], kTileBytes);
        tma_load_3d(sK + ks * kTileBytes, &tmk, &S.kfull[ks], 0, y, unit);
        tma_load_3d(sK + ks * kTileBytes + kHalfTile, &tmk, &S.kfull[ks], 64, y, unit);
        ++issued_k;
        if (i >= C::VS && !mbar_wait(&S.vempty[vs], ((i / C::VS) + 1) & 1, &S.abort)) { failed = true; break; }
        mbar_arrive_expect_tx(&S.vfull[vs], kTileBytes);
        tma_load_3d(sV + vs * kTileBytes, &tmv, &S.vfull[vs], 0, y, unit);
        tma_load_3d(sV + vs * kTileBytes + kHalfTile, &tmv, &S.vfull[vs], 64, y, unit);
        ++issued_v;
      }
      if (failed) {
        S.abort = 1;
        atomicOr(p.status, DROPKV_FLAG_TIMEOUT);
        for (int i = max(0, issued_k - C::KS); i < issued_k; ++i) mbar_drain(&S.kfull[i % C::KS], (i / C::KS) & 1);
        for (int i = max(0, issued_v - C::VS); i < issued_v; ++i) mbar_drain(&S.vfull[i % C::VS], (i / C::VS) & 1);
      }
    }
    __syncwarp();
  } else if (T > 0 && warp == 5) {
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
        const int pb = i & 1, vs = i % C::VS;
        if (!mbar_wait(&S.pfull[pb], (i >> 1) & 1, &S.abort)) { ok = false; break; }
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
  } else if (T > 0 && warp < 4) {
    // ---------------------------------------------------- softmax workers
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float lsum[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) lsum[r] = 0.f;
    for (int i = 0; i < T; ++i) {
      const int tile = t0 + i, sb = i & 1, vs = i % C::VS;
      const int j = tile * kTile + tid;
      const bool tail = tile * kTile + kTile > nb;       // tile holds slots past the sequence
      bool ok = mbar_wait(&S.sfull[sb], (i >> 1) & 1, &S.abort);
      if (ok && i >= 2) ok = mbar_wait(&S.pempty[sb], ((i >> 1) + 1) & 1, &S.abort);
      if (ok && tail) ok = mbar_wait(&S.vfull[vs], (i / C::VS) & 1, &S.abort);
      if (named_bar_or(1, kWorkers, !ok)) { failed = true; break; }
      tc_fence_after();
      float y[NR];
#pragma unroll
      for (int c0 = 0; c0 < NR; c0 += 16) tmem_ld16(tS + lane_base + sb * NR + c0, &y[c0]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.sempty[sb]);

      uint64_t vis = 0;
      bool need = false;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        y[r] *= p.scale_log2;
        const bool v_r = (j < nb) && (j <= S.pos[r]);
        vis |= (uint64_t)v_r << r;
        need |= v_r && (y[r] - S.mref[r] > kRescaleLog2);
      }
      if (named_bar_or(1, kWorkers, need)) {
        // new reference = max(old reference, this tile's max) per row
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float v = ((vis >> r) & 1) ? y[r] : -INFINITY;
          const uint32_t u = __reduce_max_sync(0xffffffffu, f2ord(v));
          if (lane == 0) S.red[warp][r] = ord2f(u);
        }
        named_bar(2, kWorkers);                 // per-warp maxima complete
        float factor[NR];
        float my_ref = 0.f;                     // new reference of row `tid` (tid < NR)
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float old = S.mref[r];
          const float nm = fmaxf(fmaxf(fmaxf(S.red[0][r], S.red[1][r]), fmaxf(S.red[2][r], S.red[3][r])), old);
          factor[r] = (old == -INFINITY) ? 0.f : exp2f(old - nm);
          lsum[r] *= factor[r];
          if (r == tid) my_ref = nm;
        }
        if (i > 0) {
          // rescale the accumulated O (lane = head dimension) once PV of tile i-1 is done
          const bool okw = mbar_wait(&S.ofull, (i - 1) & 1, &S.abort);
          if (named_bar_or(2, kWorkers, !okw)) { failed = true; break; }
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < NR; c0 += 16) {
            float o[16];
            tmem_ld16(tO + lane_base + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 16; ++q) o[q] *= factor[c0 + q];
            tmem_st16(tO + lane_base + c0, o);
          }
          tmem_wait_st();
          tc_fence_before();
        }
        named_bar(2, kWorkers);                 // every thread has read the old references
        if (tid < NR) S.mref[tid] = my_ref;
        named_bar(2, kWorkers);                 // new references visible
      }
      // exponentials relative to the row reference, split into bf16 hi + lo
      uint8_t* phi = sP + (sb * 2 + 0) * C::kPBytes;
      uint8_t* plo = sP + (sb * 2 + 1) * C::kPBytes;
#pragma unroll
      for (int r8 = 0; r8 < NR / 8; ++r8) {
        uint32_t hp[4], lp[4];
#pragma unroll
        for (int q = 0; q < 8; q += 2) {
          float e2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int r = r8 * 8 + q + u;
            const float e = ((vis >> r) & 1) ? exp2f(y[r] - S.mref[r]) : 0.f;
            lsum[r] += e;
            e2[u] = e;
          }
          const __nv_bfloat16 h0 = __float2bfloat16_rn(e2[0]), h1 = __float2bfloat16_rn(e2[1]);
          const __nv_bfloat16 l0 = __float2bfloat16_rn(e2[0] - __bfloat162float(h0));
          const __nv_bfloat16 l1 = __float2bfloat16_rn(e2[1] - __bfloat162float(h1));
          hp[q >> 1] = pack_bf16x2(h0, h1);
          lp[q >> 1] = pack_bf16x2(l0, l1);
        }
        const uint32_t off = interleave_mn_offset(tid, r8 * 8, NR);
        *reinterpret_cast<uint4*>(phi + off) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
        *reinterpret_cast<uint4*>(plo + off) = make_uint4(lp[0], lp[1], lp[2], lp[3]);
      }
      if (tail && j >= nb) {
        // slots past the sequence may hold anything (NaN): zero their V rows
        // so that 0 * NaN never reaches the PV accumulator
        uint8_t* vrow = sV + vs * kTileBytes + tid * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vrow + kHalfTile + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pfull[sb]);
    }
    // ------------------------------------------------ partial state of this split
    bool okw = true;
    if (!failed) okw = mbar_wait(&S.ofull, (T - 1) & 1, &S.abort);
    if (named_bar_or(1, kWorkers, failed || !okw)) failed = true;
    const size_t part = (size_t)unit * p.splits + split;
    if (!failed) {
      tc_fence_after();
      float* po = p.part_o + part * R * p.d;
#pragma unroll
      for (int c0 = 0; c0 < NR; c0 += 16) {
        float o[16];
        tmem_ld16(tO + lane_base + c0, o);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q)
          if (c0 + q < R && tid < p.d) po[(size_t)(c0 + q) * p.d + tid] = o[q];
      }
      tc_fence_before();
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float v = warp_sum(lsum[r]);
      if (lane == 0) S.red[warp][r] = v;
    }
    named_bar(2, kWorkers);
    if (tid < R) {
      float* ml = p.part_ml + (part * R + tid) * 2;
      ml[0] = S.mref[tid];
      ml[1] = failed ? 0.f : (S.red[0][tid] + S.red[1][tid]) + (S.red[2][tid] + S.red[3][tid]);
    }
  }

  if (T == 0) {
    // empty split (past the end of a shorter sequence): publish an empty state
    const size_t part = (size_t)unit * p.splits + split;
    for (int idx = tid; idx < R; idx += kThreads) {
      p.part_ml[(part * R + idx) * 2] = -INFINITY;
      p.part_ml[(part * R + idx) * 2 + 1] = 0.f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (T > 0 && warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  // ---------------------------------------------------- split-K merge ticket
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t t = atomicAdd(&p.tickets[unit], 1u);
    S.is_last = (t == (uint32_t)p.splits - 1);
  }
  __syncthreads();
  if (S.is_last) {
    __threadfence();
    float* wts = reinterpret_cast<float*>(sK);                     // [splits][R]
    float* Ms = wts + (size_t)p.splits * R;
    float* Ls = Ms + kMaxR;
    merge_unit(p, unit, wts, Ms, Ls, tid);
    if (tid == 0) p.tickets[unit] = 0;
  }
}

// ============================================================== pass 2
template <int NR>
struct Pass2Cfg {
  static constexpr int KS = 3;
  static constexpr int VS = NR <= 32 ? 3 : 2;
  static constexpr int kQBytes = NR * kDPad * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + KS * kTileBytes;
  static constexpr int kOffQ = kOffV + VS * kTileBytes;
  static constexpr int kOffAhi = kOffQ + kQBytes;
  static constexpr int kOffAlo = kOffAhi + kQBytes;
  static constexpr int kOffSmall = kOffAlo + kQBytes;
  static constexpr uint32_t kTmemCols = (4 * NR <= 64) ? 64u : (4 * NR <= 128 ? 128u : 256u);
};

struct Pass2Small {
  uint64_t kfull[3], kempty[3], vfull[3], vempty[3];
  uint64_t accfull[2], accempty[2], drain;
  uint32_t tmem_base;
  int abort;
  int pos[kMaxR];
  float m2[kMaxR], L[kMaxR], aa[kMaxR];
};

template <int NR>
constexpr int pass2_smem_bytes() {
  return Pass2Cfg<NR>::kOffSmall + (int)sizeof(Pass2Small) + 1024;
}

template <int NR>
__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                 const AttnParams p) {
  using C = Pass2Cfg<NR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sK = sm + C::kOffK;
  uint8_t* sV = sm + C::kOffV;
  uint8_t* sQ = sm + C::kOffQ;
  uint8_t* sAhi = sm + C::kOffAhi;
  uint8_t* sAlo = sm + C::kOffAlo;
  Pass2Small& S = *reinterpret_cast<Pass2Small*>(sm + C::kOffSmall);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, unit = blockIdx.y;
  const int b = unit / p.Hkv, h = unit - b * p.Hkv;
  const int nb = p.lengths ? p.lengths[b] : p.n_max;
  if (nb < p.w || nb > p.n_max) return;      // flagged by pass 1
  const int R = p.R;
  const int t0 = split * p.tpc;
  const int t1 = min(t0 + p.tpc, ceil_div(nb, kTile));
  const int T = t1 - t0;
  if (T <= 0) return;

  if (tid == 0) {
    for (int i = 0; i < C::KS; ++i) { mbar_init(&S.kfull[i], 1); mbar_init(&S.kempty[i], 1); }
    for (int i = 0; i < C::VS; ++i) { mbar_init(&S.vfull[i], 1); mbar_init(&S.vempty[i], 5); }
    for (int i = 0; i < 2; ++i) { mbar_init(&S.accfull[i], 1); mbar_init(&S.accempty[i], 4); }
    mbar_init(&S.drain, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(&S.tmem_base, C::kTmemCols);
  if (tid < kWorkers) {
    const __nv_bfloat16* qsrc = p.q + ((size_t)b * p.Hq + (size_t)h * p.g) * p.w * p.d;
    stage_rows_sw128(sQ, qsrc, NR, R, p.d, p.d, tid, kWorkers);
    const __nv_bfloat16* ahl = p.ahl + (size_t)unit * 2 * kMaxR * kDPad;
    stage_rows_sw128(sAhi, ahl, NR, NR, kDPad, kDPad, tid, kWorkers);
    stage_rows_sw128(sAlo, ahl + kMaxR * kDPad, NR, NR, kDPad, kDPad, tid, kWorkers);
    fence_proxy_async_smem();
    if (tid < kMaxR) {
      const bool real = tid < R;
      S.pos[tid] = real ? nb - p.w + (tid % p.w) : -1;
      const size_t o = (size_t)unit * R + tid;
      S.m2[tid] = real ? p.m2[o] : 0.f;
      S.L[tid] = real ? p.l[o] : 1.f;
      S.aa[tid] = real ? p.aa[o] : 0.f;
    }
  }
  if (warp == 4 && lane == 0) { tma_prefetch_desc(&tmk); tma_prefetch_desc(&tmv); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  bool failed = false;

  if (warp == 4) {
    if (lane == 0) {
      int issued_k = 0, issued_v = 0;
      for (int i = 0; i < T; ++i) {
        const int y = (t0 + i) * kTile;
        const int ks = i % C::KS, vs = i % C::VS;
        if (i >= C::KS && !mbar_wait(&S.kempty[ks], ((i / C::KS) + 1) & 1, &S.abort)) { failed = true; break; }
        mbar_arrive_expect_tx(&S.kfull[ks], kTileBytes);
        tma_load_3d(sK + ks * kTileBytes, &tmk, &S.kfull[ks], 0, y, unit);
        tma_load_3d(sK + ks * kTileBytes + kHalfTile, &tmk, &S.kfull[ks], 64, y, unit);
        ++issued_k;
        if (i >= C::VS && !mbar_wait(&S.vempty[vs], ((i / C::VS) + 1) & 1, &S.abort)) { failed = true; break; }
        mbar_arrive_expect_tx(&S.vfull[vs], kTileBytes);
        tma_load_3d(sV + vs * kTileBytes, &tmv, &S.vfull[vs], 0, y, unit);
        tma_load_3d(sV + vs * kTileBytes + kHalfTile, &tmv, &S.vfull[vs], 64, y, unit);
        ++issued_v;
      }
      if (failed) {
        S.abort = 1;
        atomicOr(p.status, DROPKV_FLAG_TIMEOUT);
        for (int i = max(0, issued_k - C::KS); i < issued_k; ++i) mbar_drain(&S.kfull[i % C::KS], (i / C::KS) & 1);
        for (int i = max(0, issued_v - C::VS); i < issued_v; ++i) mbar_drain(&S.vfull[i % C::VS], (i / C::VS) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t idS = umma_idesc_bf16(128, NR, 0, 0);
      const uint32_t qaddr = smem_addr(sQ), ahi = smem_addr(sAhi), alo = smem_addr(sAlo);
      bool ok = true;
      for (int i = 0; i < T; ++i) {
        const int ks = i % C::KS, vs = i % C::VS, ab = i & 1;
        const uint32_t dS = tmem + ab * 2 * NR, dAV = dS + NR;
        if (!mbar_wait(&S.kfull[ks], (i / C::KS) & 1, &S.abort)) { ok = false; break; }
        if (i >= 2 && !mbar_wait(&S.accempty[ab], ((i >> 1) + 1) & 1, &S.abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kb = smem_addr(sK + ks * kTileBytes);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_bf16(dS, desc_kmajor_sw128(kb, kTile, s), desc_kmajor_sw128(qaddr, NR, s), idS, s > 0);
        umma_commit(&S.kempty[ks]);
        if (!mbar_wait(&S.vfull[vs], (i / C::VS) & 1, &S.abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vb = smem_addr(sV + vs * kTileBytes);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_bf16(dAV, desc_kmajor_sw128(vb, kTile, s), desc_kmajor_sw128(ahi, NR, s), idS, s > 0);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_bf16(dAV, desc_kmajor_sw128(vb, kTile, s), desc_kmajor_sw128(alo, NR, s), idS, 1);
        umma_commit(&S.vempty[vs]);
        umma_commit(&S.accfull[ab]);
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
  } else {
    // ---------------------------------------------------- score workers
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float inv_g = 1.0f / (float)p.g;
    float* raw = p.raw + (size_t)unit * p.n_max;
    uint32_t flags = 0;
    for (int i = 0; i < T; ++i) {
      const int tile = t0 + i, vs = i % C::VS, ab = i & 1;
      const int j = tile * kTile + tid;
      // |v_j|^2 from the staged V row (order of the 128 columns is irrelevant)
      bool ok = mbar_wait(&S.vfull[vs], (i / C::VS) & 1, &S.abort);
      float vv = 0.f;
      if (ok) {
        const uint8_t* vrow = sV + vs * kTileBytes + tid * 128;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint4 raw4 = *reinterpret_cast<const uint4*>(vrow + (c >> 3) * kHalfTile + (c & 7) * 16);
          const uint32_t w4[4] = {raw4.x, raw4.y, raw4.z, raw4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float lo = __uint_as_float(w4[u] << 16), hi = __uint_as_float(w4[u] & 0xFFFF0000u);
            vv = fmaf(lo, lo, vv);
            vv = fmaf(hi, hi, vv);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.vempty[vs]);
      if (ok) ok = mbar_wait(&S.accfull[ab], (i >> 1) & 1, &S.abort);
      if (!ok) { failed = true; break; }      // no named barriers in this role: exit per thread
      tc_fence_after();
      float sv[NR], av[NR];
#pragma unroll
      for (int c0 = 0; c0 < NR; c0 += 16) {
        tmem_ld16(tmem + lane_base + ab * 2 * NR + c0, &sv[c0]);
        tmem_ld16(tmem + lane_base + ab * 2 * NR + NR + c0, &av[c0]);
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.accempty[ab]);
      if (j < nb) {
        float s = 0.f;
        bool singular = false;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          if (j <= S.pos[r]) {
            const float e = exp2f(sv[r] * p.scale_log2 - S.m2[r]);
            const float den = S.L[r] - e;           // l (1 - p_j)
            if (!(den > 0.f)) singular = true;
            const float ratio = __fdividef(e, den);  // p_j / (1 - p_j)
            const float dist = fmaxf(fmaf(-2.f, av[r], S.aa[r] + vv), 0.f);   // |a - v_j|^2
            s = fmaf(ratio * ratio, dist, s);
          }
        }
        s *= inv_g;
        if (singular) {
          s = INFINITY;
          flags |= DROPKV_FLAG_SINGULAR;
        } else if (!isfinite(s)) {
          flags |= DROPKV_FLAG_NONFINITE;
        }
        raw[j] = s;
      }
    }
    if (flags) atomicOr(p.status, flags);
  }
  if (failed) S.abort = 1;
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int NR>
cudaError_t launch_pass1_t(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  constexpr int smem = pass1_smem_bytes<NR>();
  static_assert(smem <= 232448, "pass-1 shared memory exceeds the per-CTA limit");
  cudaError_t e = cudaFuncSetAttribute(window_attention_kernel<NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  window_attention_kernel<NR><<<dim3(p.splits, p.U), kThreads, smem, st>>>(tk, tv, p);
  return cudaGetLastError();
}

template <int NR>
cudaError_t launch_pass2_t(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  constexpr int smem = pass2_smem_bytes<NR>();
  static_assert(smem <= 232448, "pass-2 shared memory exceeds the per-CTA limit");
  cudaError_t e = cudaFuncSetAttribute(score_kernel<NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  score_kernel<NR><<<dim3(p.splits, p.U), kThreads, smem, st>>>(tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_window_attention(const AttnParams& p, int NR, const CUtensorMap& tk, const CUtensorMap& tv,
                                    int, cudaStream_t st) {
  switch (NR) {
    case 16: return launch_pass1_t<16>(p, tk, tv, st);
    case 32: return launch_pass1_t<32>(p, tk, tv, st);
    case 64: return launch_pass1_t<64>(p, tk, tv, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_score(const AttnParams& p, int NR, const CUtensorMap& tk, const CUtensorMap& tv,
                         cudaStream_t st) {
  switch (NR) {
    case 16: return launch_pass2_t<16>(p, tk, tv, st);
    case 32: return launch_pass2_t<32>(p, tk, tv, st);
    case 64: return launch_pass2_t<64>(p, tk, tv, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dropkv
