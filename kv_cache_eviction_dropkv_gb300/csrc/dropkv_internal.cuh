// Internal declarations shared by the library's translation units: problem
// geometry, the workspace plan, kernel parameter blocks and launchers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/dropkv.h"

namespace dropkv {

constexpr int kTile = 128;          // tokens per K/V tile (the MMA M dimension)
constexpr int kDPad = 128;          // head dimension as staged in shared memory
constexpr int kMaxR = 64;           // rows (g * w) per KV head supported
constexpr int kMaxSplits = 160;    // split-K partial states per KV head (merge holds 5 per lane)
constexpr int kSelChunk = 16384;    // tokens per block in the selection kernels
constexpr int kLayerChunk = 4096;   // tokens per block in the layer-wide selection kernels
constexpr int kHistBins = 4096;     // first-level radix histogram (top 12 key bits)
constexpr int kCandCap = 8192;      // candidates resolved in shared memory
constexpr int kMaxPool = 63;

// Geometry derived from dropkv_shape.
struct Geom {
  int B, Hq, Hkv, d, n_max, w;
  int g, R, NR;          // NR: R rounded up to the MMA width instantiated (16, 32 or 64)
  int U;                 // B * Hkv units (KV heads)
  int tiles_max;         // ceil(n_max / kTile)
  int ctas;              // CTAs of a pass grid: max(U, SMs), below 256 when above U
  int even;              // CTAs per unit when all units have one length
  int splits1;           // pass-1 partial slots per unit (most CTAs a unit can get)
  int splits2;           // most pass-2 CTAs a unit can get
  int chunks;            // ceil(n_max / kSelChunk)
  int layer_chunks;      // ceil(n_max / kLayerChunk)
};

// Byte offsets of the workspace regions (all 256-byte aligned).
struct WsPlan {
  size_t m, l, a;                // exported statistics (see dropkv.h)
  size_t m2;                     // max in log2 units
  size_t aa;                     // K = |a'|^2 + 2 a'.c per row
  size_t ahl;                    // bf16 [U][2][64][128]: a' = a - c split into hi + lo parts
  size_t cvec, cflag;            // f32 [U][128] shift c of each head, i32 [U] 1 when shifted
  size_t dom_s, dom_l;           // dominated rows: pass-1 split of the dominant key, L of the other splits
  size_t dom_o;                  // dominated rows: f32 [U][R][d] sum of the other splits' O
  size_t part_o, part_ml;        // pass-1 partial states (part_ml: m, l, largest logit, unused)
  size_t tile_ctr;               // u32 [U]: pass-2 tile claims (cleared by the merge kernel)
  size_t qwin;                   // bf16 [B][Hq][w][d]: the window query rows (prefilled path)
  size_t raw;                    // f32 [U][n_max] raw scores when the caller passes none
  // selection
  size_t hist;                   // u32 [U][kHistBins]
  size_t hist2;                  // u32 [U][kHistBins] (second level)
  size_t sel_state;              // u32 [U][8]
  size_t cand;                   // u32 [U][kCandCap][2]
  size_t cand_cnt;               // u32 [U]
  size_t sel_tickets;            // u32 [U][2]
  size_t chunk_kept;             // u32 [U][chunks]
  size_t chunk_off;              // u32 [U][chunks]
  size_t layer_zero_begin;       // layer-wide selection: h1, h2 [B][4096], h3 [B][256] (cleared per call)
  size_t layer_h1, layer_h2, layer_h3;
  size_t layer_zero_end;
  size_t layer_state;            // u32 [B][8]
  size_t layer_counts;           // u32 [B][Hkv][chunks][2]
  size_t sel_zero_begin, sel_zero_end;   // range cleared at the start of dropkv_select
  size_t total;
};

bool make_geom(const dropkv_shape* s, int num_sms, Geom* g);
WsPlan make_plan(const Geom& g);

// Parameter block of the two attention passes.
// Score kinds (DROPKV_SCORE_* of the C ABI).
constexpr int kKindDropKV = 0;   // exact single-token output perturbation
constexpr int kKindSnapKV = 1;   // window sum of attention probabilities

// A window row is "dominated" when its largest attention probability reaches
// kDomP: then 1 - p of that key and |a - v| are tiny differences of large
// quantities, and pass 2 takes that key's score from the attention output
// recomputed without it (see the pass-2 kernel).
constexpr float kDomP = 0.8f;

struct AttnParams {
  const __nv_bfloat16* q;        // [B][Hq][w][d]
  const __nv_bfloat16* v;        // [B][Hkv][n_max][d] (pass 2 reads the rows of dominant keys)
  const int32_t* lengths;        // [B] or null
  int B, Hq, Hkv, d, n_max, w, g, R, U;
  int NR;                        // R rounded up to the MMA width (16, 32 or 64)
  int splits;                    // most CTAs per unit (pass 1: its partial slots per unit)
  int splits1;                   // pass-1 partial slots per unit (both passes)
  int ctas;                      // CTAs of the pass grid (>= U)
  int even;                      // > 0: every unit gets this many CTAs; 0: shares by length
  float scale_log2;              // log2(e) / sqrt(d)
  // workspace
  float *m, *l, *a, *m2;
  float* aa;                     // [U][R] K = |a'|^2 + 2 a'.c
  __nv_bfloat16* ahl;            // [U][2][64][128] a' split into bf16 hi, then lo (rows past R zero)
  float* cvec;                   // [U][128] shift c (bf16 values; zero when not shifted)
  int* cflag;                    // [U] 1: the head's scores use the shift
  int* dom_s;                    // [U][R] pass-1 split holding a dominated row's largest probability, else -1
  float* dom_l;                  // [U][R] normaliser of the other splits (dominated rows)
  float* dom_o;                  // [U][R][d] unnormalised output of the other splits (dominated rows)
  float *part_o, *part_ml;
  uint32_t* tile_ctr;            // [U] next unclaimed pass-2 tile of each KV head
  float* raw;                    // raw score output [U][n_max]
  uint32_t* status;
  int kind;                      // kKindDropKV or kKindSnapKV
  int part_splits;               // > 0: partial states per unit when they come from the prefill kernel (1)
};

// The prefill kernel (a causal attention over every query row, the window
// states a by-product) in pass 1's place.
struct PrefillParams {
  const __nv_bfloat16* q;        // [B][Hq][n_max][d] every query row
  __nv_bfloat16* out;            // [B][Hq][n_max][d] attention output (rows < n_b written)
  __nv_bfloat16* q_win;          // [B][Hq][w][d] the window rows of q (pass 2's q)
  const int32_t* lengths;        // [B] or null
  float *part_o, *part_ml;       // window rows' states in pass 1's layout (one partial per row)
  int B, Hq, Hkv, g, d, n_max, w, R, splits;
  float scale_log2;
  uint32_t* status;
};

struct PoolParams {
  const float* raw;
  float* scores;
  const int32_t* lengths;
  int B, Hkv, n_max, w, half, protect;
  uint32_t* status;
};

struct SelParams {
  const float* scores;
  const int32_t* lengths;
  const int32_t* evict_k;
  int32_t* kept_idx;
  int32_t* kept_len;
  int B, Hkv, n_max, protect, chunks;
  uint32_t *hist, *hist2, *state, *cand, *cand_cnt, *tickets, *chunk_kept, *chunk_off;
  uint32_t* status;
  // Optional pooling stage (pool.raw != nullptr): the selection first pools
  // pool.raw into pool.scores (== scores) as pool_protect_kernel would.
  PoolParams pool;
};

struct CompactParams {
  const uint8_t* k;
  const uint8_t* v;
  const int32_t* kept_idx;
  const int32_t* kept_len;
  uint8_t* k_out;
  uint8_t* v_out;
  int B, Hkv, n_max, row_bytes, out_rows;
  uint32_t* status;
  int per_head;                  // kept_len is [B][Hkv] (layer-wide selection), else [B]
};

// Layer-wide selection: one pool per sequence over all its KV heads.
struct LayerSelParams {
  const float* scores;           // [B][Hkv][n_max]
  const int32_t* lengths;        // [B] or null
  const int32_t* evict_total;    // [B]
  int32_t* kept_idx;             // [B][Hkv][n_max]
  int32_t* kept_len;             // [B][Hkv]
  int B, Hkv, n_max, protect, chunks;   // chunks per head
  uint32_t *h1, *h2, *h3;        // [B][4096], [B][4096], [B][256] (cleared before the first kernel)
  uint32_t* state;               // [B][8]
  uint32_t* counts;              // [B][Hkv][chunks][2]: slots above T, slots equal to T
                                 // (chunks of kLayerChunk slots)
  uint32_t* status;
};

// Launch with programmatic dependent launch: the kernel may be scheduled
// while its predecessor in the stream is finishing.  Every kernel of the
// library calls grid_dep_wait() before it reads anything an earlier kernel
// wrote and before its first global write, so stream order is preserved.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Steps S1-S4 on the caller's workspace (the body of dropkv_score and its
// variants).  scoring_regions_only: the workspace need only hold the regions
// scoring uses (the ones ahead of the selection's).
// Inputs of the prefilled path: every query row and the attention output.
struct PrefillIn {
  const void* q;                 // bf16 [B][Hq][n_max][d]
  void* out;                     // bf16 [B][Hq][n_max][d]
};

dropkv_status score_core(const dropkv_shape* shape, const void* q_window, const void* k, const void* v,
                         const int32_t* lengths, int32_t pool_kernel, int32_t protect, float* scores,
                         float* raw_scores, void* workspace, size_t workspace_bytes, uint32_t* status,
                         cudaStream_t stream, cudaEvent_t* ev, PoolParams* defer_pool, int kind,
                         bool scoring_regions_only, const PrefillIn* pre = nullptr);

cudaError_t launch_window_attention(const AttnParams& p, int NR, const CUtensorMap& tk, const CUtensorMap& tv,
                                    int num_ctas_x, cudaStream_t st);
cudaError_t launch_merge(const AttnParams& p, cudaStream_t st);
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t st);
cudaError_t launch_score(const AttnParams& p, int NR, const CUtensorMap& tk, const CUtensorMap& tv,
                         cudaStream_t st);
cudaError_t launch_pool_protect(const PoolParams& p, cudaStream_t st);
cudaError_t launch_select(const SelParams& p, size_t zero_bytes, void* zero_base, cudaStream_t st);
cudaError_t launch_select_layer(const LayerSelParams& p, size_t zero_bytes, void* zero_base, cudaStream_t st);
cudaError_t launch_compact(const CompactParams& p, cudaStream_t st);

}  // namespace dropkv
