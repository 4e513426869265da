/*
 * dropkv.h -- C ABI of the GB300 (sm_103a) DropKV eviction-scoring path.
 *
 * The method ("DropKV: Decoupling Residual-Output Perturbation for Near-Optimal
 * KV-Cache Eviction"; "DropKV: Exact single-entry output-perturbation scoring",
 * Core equation and Algorithm 1 summary): for every KV head, the last w prompt
 * queries of each query head in its GQA group attend causally, tail-aligned,
 * over the n cached keys; with p = softmax(K q / sqrt(d)) and a = sum_j p_j v_j,
 * each cached token j is scored by its exact single-token output perturbation
 * s_j = sum_t || p_j / (1 - p_j) (a - v_j) ||^2 ; scores are averaged over the
 * query heads of the group, max-pooled along the sequence, the last slots are
 * protected (+inf), the k lowest are evicted and the kept K/V rows compacted.
 *
 * Conventions (all entry points):
 *  - Every buffer is owned by the caller.  Pointers marked "device" are CUDA
 *    device pointers, 16-byte aligned, densely packed in the stated layout.
 *    The library allocates no device memory.
 *  - Calls are asynchronous on `stream` (any CUDA stream of the current
 *    device; 0 = the legacy default stream).  A host-detectable error returns
 *    immediately with nothing launched.
 *  - Errors found on the device (a singular or non-finite score, an invalid
 *    length or eviction count, a pipeline wait that timed out) are OR-ed into
 *    the caller's 32-bit device status word (`status`, zeroed by the caller
 *    before the first call); the call still completes and writes defined
 *    values.  dropkv_read_status() syncs the stream and reports the word.
 *  - bf16 inputs are read as stored; arithmetic is fp32 with bf16 operands on
 *    the tensor cores and fp32 accumulation.
 */
#ifndef DROPKV_H
#define DROPKV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define DROPKV_API __attribute__((visibility("default")))
#else
#define DROPKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DROPKV_OK = 0,
  DROPKV_ERR_INVALID_ARG = 1,   /* bad shape, pointer, alignment, kernel size or aliasing */
  DROPKV_ERR_WORKSPACE = 2,     /* workspace missing or smaller than dropkv_workspace_size() */
  DROPKV_ERR_SINGULAR = 3,      /* some p_j rounded to 1: exact removal is singular (rejected, no epsilon) */
  DROPKV_ERR_NONFINITE = 4,     /* a score or attention statistic is not finite */
  DROPKV_ERR_CUDA = 5,          /* a CUDA runtime call failed */
  DROPKV_ERR_UNSUPPORTED = 6,   /* shape outside the supported range (see dropkv_shape) */
  DROPKV_ERR_DEVICE_ARG = 7,    /* device-side argument check failed (lengths, eviction counts, capacity) */
  DROPKV_ERR_TIMEOUT = 8        /* a kernel pipeline wait gave up (flag set instead of hanging) */
} dropkv_status;

/* Bits of the device status word. */
#define DROPKV_FLAG_SINGULAR   0x01u
#define DROPKV_FLAG_NONFINITE  0x02u
#define DROPKV_FLAG_BAD_LENGTH 0x04u   /* lengths[b] outside [w, n_max] (or < protect) */
#define DROPKV_FLAG_BAD_K      0x08u   /* evict_k[b] outside [0, n_b - protect] (evict_total[b]
                                          outside [0, Hkv (n_b - protect)] for the layer-wide call) */
#define DROPKV_FLAG_OVERFLOW   0x10u   /* a kept count > out_rows in a compaction */
#define DROPKV_FLAG_TIMEOUT    0x20u
#define DROPKV_FLAG_INTERNAL   0x40u   /* a selection consistency check failed (kept count != n_b - k_b) */
/* Detail bits that accompany DROPKV_FLAG_NONFINITE: where the value appeared. */
#define DROPKV_FLAG_NONFINITE_STATS 0x100u  /* window statistics (normaliser or |a|^2) */
#define DROPKV_FLAG_NONFINITE_SCORE 0x200u  /* a token score */

/* Score kinds of dropkv_score_ex / dropkv_evict_ex. */
#define DROPKV_SCORE_DROPKV 0   /* s_j = sum_t ||p_j / (1 - p_j) (a - v_j)||^2 (the method) */
#define DROPKV_SCORE_SNAPKV 1   /* s_j = sum_t p_j: the attention-only baseline ("DropKV: Decoupling ...",
                                 * Appendix B, Table 14, SnapKV row), same window, GQA mean,
                                 * pooling, protection, selection and compaction; reads K only */

/* Problem shape.  Supported: B >= 1; Hq % Hkv == 0; g = Hq / Hkv; R = g * w <= 64;
 * d a multiple of 8 in [8, 128]; 1 <= w <= n_max < 2^31. */
typedef struct {
  int32_t B;       /* batch (sequences) */
  int32_t Hq;      /* query heads */
  int32_t Hkv;     /* KV heads */
  int32_t d;       /* head dimension */
  int32_t n_max;   /* cache capacity per sequence (padded length) */
  int32_t w;       /* observation window: tail queries per query head */
} dropkv_shape;

/* Infrastructure (no passage of the pages): the workspace sizing of this
 * library's own scratch layout.
 * Bytes of device workspace the calls that take one need for `shape` on the
 * current device (0 if the shape is invalid or unsupported, or no device is
 * present).  One workspace serves every call on that shape (not two calls at
 * once: calls that overlap on the GPU must use separate workspaces).  After
 * dropkv_score completes, the workspace starts with the window statistics of
 * step S1 (U = B * Hkv, R = g * w, row r = h_local * w + t of KV head (b, h),
 * logits x_j = q.k_j / sqrt(d) over the keys the row sees):
 *   float lse[U][R]    log sum_j exp(x_j)        (offset 0)
 *   float a[U][R][d]   sum_j p_j v_j             (offset round_up(4*U*R, 256)) */
DROPKV_API size_t dropkv_workspace_size(const dropkv_shape* shape);

/* Steps S1-S4: window attention with its split-K merge, per-token
 * perturbation score with the GQA average, MaxPool1D and recent-slot
 * protection.
 *   q_window  device bf16 [B][Hq][w][d]  last w query rows of every query head
 *   k, v      device bf16 [B][Hkv][n_max][d]  cached keys / values; only rows
 *             j < lengths[b] are read
 *   lengths   device int32 [B] (n_b), or NULL for n_b = n_max
 *   pool_kernel  odd, 1..63: MaxPool1D kernel (stride 1, window clipped to [0, n_b))
 *   protect   >= 0: slots j >= n_b - protect get +inf after pooling
 *   scores    device float [B][Hkv][n_max]: final score of slot j < n_b
 *             (slots >= n_b are not written)
 *   raw_scores  device float [B][Hkv][n_max] or NULL: GQA-averaged score
 *             before pooling
 *   workspace / workspace_bytes  device scratch of dropkv_workspace_size() bytes
 *   status    device uint32 status word
 * Numerics (fp32 with bf16 tensor-core operands):
 *  - A key with p_j <= 1/2 is scored as e/(L - e) (a - v).  A row whose
 *    largest key holds about 0.8 of its mass or more (judged by the merge
 *    from bf16 maxima) is "dominated": that key's term is taken in the equal
 *    form p*^2 |a_rest - v*|^2, with the other keys' mass L_rest and output
 *    summed on their own (no cancellation as p* -> 1), by the CTA that holds
 *    the key.  The key is rejected as singular (DROPKV_FLAG_SINGULAR, score
 *    +inf) when L_rest <= 2^-53 e*, i.e. when p* rounds to 1 in double
 *    precision, the oracle's rule.
 *  - |a - v_j|^2 is expanded around c: K - 2 a'.v_j + |v_j - c|^2 with
 *    a' = a - c and K = |a'|^2 + 2 a'.c.  c is window row 0's output over the
 *    keys of the first pass-1 split, rounded to bf16, when |c|^2 > 2d (values
 *    sharing a large offset), else 0.
 * Sources: "... output-perturbation scoring", Core equation, Algorithm 1
 * summary, Code mapping (tail-aligned causality, GQA). */
DROPKV_API dropkv_status dropkv_score(const dropkv_shape* shape, const void* q_window, const void* k, const void* v,
                           const int32_t* lengths, int32_t pool_kernel, int32_t protect, float* scores,
                           float* raw_scores, void* workspace, size_t workspace_bytes, uint32_t* status,
                           cudaStream_t stream);

/* The prompt's causal attention alone (the kernel of dropkv_evict_prefill
 * without the eviction): attn_out[b][hq][i] = softmax over keys j <= i of
 * q_i k_j / sqrt(d), times v, for every row i < n_b ("DropKV: Decoupling ...",
 * section 2.1).  q, k, v, attn_out as in dropkv_evict_prefill; the workspace
 * (dropkv_workspace_size bytes) receives the window states as a by-product.
 * For comparison with the fused call: this followed by dropkv_evict reads K
 * and V once more in pass 1. */
DROPKV_API dropkv_status dropkv_prefill_attention(const dropkv_shape* shape, const void* q, const void* k,
                                                  const void* v, const int32_t* lengths, void* attn_out,
                                                  void* workspace, size_t workspace_bytes, uint32_t* status,
                                                  cudaStream_t stream);

/* Steps S1-S6 fused into the model's prefill attention: a causal attention
 * over every query row of the prompt ("DropKV: Decoupling ...", section 2.1;
 * the scorer fused into prefill, sections 1 and 5.4) writes the attention
 * output and, as a by-product of its last w rows, the window statistics that
 * step S1 would compute; the eviction then runs without pass 1's read of K
 * and V: merge, scoring, pooling, selection and compaction as dropkv_evict_ex.
 *   q         device bf16 [B][Hq][n_max][d]: every query row of the prompt (row
 *             i of head hq attends to keys j <= i of KV head hq / g)
 *   attn_out  device bf16 [B][Hq][n_max][d]: softmax(q k^T / sqrt(d)) v per row;
 *             rows >= n_b are not written; must not overlap q, k or v
 *   every other argument as dropkv_evict_ex (the window of the scores is the
 *   last w rows of q).  Window rows use P in bf16 hi + lo on the tensor cores
 *   (their statistics match pass 1's precision); the other rows use bf16 P.
 *   The window states come as one partial per row, so a KV head with a
 *   dominated row is scored by one CTA in the dominant mode (exact, slower).
 * Sources: "DropKV: Decoupling ...", sections 1, 2.1 and 5.4 (fusion into
 * prefill); "... output-perturbation scoring", Core equation. */
DROPKV_API dropkv_status dropkv_evict_prefill(const dropkv_shape* shape, int32_t score_kind, const void* q,
                                              const void* k, const void* v, const int32_t* lengths,
                                              const int32_t* evict_k, int32_t pool_kernel, int32_t protect,
                                              void* attn_out, float* scores, float* raw_scores, int32_t* kept_idx,
                                              int32_t* kept_len, int32_t out_rows, void* k_out, void* v_out,
                                              void* workspace, size_t workspace_bytes, uint32_t* status,
                                              cudaStream_t stream);

/* Infrastructure (no passage of the pages): per-kernel timing.
 * dropkv_score_ex that also records phase_events[0..4] on `stream`: before
 * pass 1 (window attention), between pass 1 and the split-K merge, between the
 * merge and pass 2 (scoring), between pass 2 and pooling, and after pooling --
 * for per-kernel timing with CUDA events.  The events are created by the
 * caller; everything else is as dropkv_score_ex. */
DROPKV_API dropkv_status dropkv_score_timed(const dropkv_shape* shape, int32_t score_kind, const void* q_window,
                                            const void* k, const void* v, const int32_t* lengths,
                                            int32_t pool_kernel, int32_t protect, float* scores, float* raw_scores,
                                            void* workspace, size_t workspace_bytes, uint32_t* status,
                                            cudaStream_t stream, cudaEvent_t* phase_events);

/* dropkv_score without a workspace argument, for callers that cannot allocate
 * device memory when they score (a host framework that owns all device memory
 * through its own pool, or a serving loop that forbids allocations after
 * start-up).  The paper has no counterpart: this is a deployment variant.
 *   Scratch: a fixed 16 MiB device array inside the library (held by every GPU
 *   that loads it until exit), enough for the scoring scratch of every shape
 *   whose dropkv_workspace_size() scoring part fits (for example B=1, Hkv=8,
 *   n=128K).  Larger shapes return DROPKV_ERR_WORKSPACE and launch nothing.
 *   Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library call.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.
 *   All calls share the array and it keeps the last call's contents: calls
 *   that overlap on the GPU (concurrent streams, other threads) race and must
 *   be serialised by the caller.  The window statistics are not exported.
 * Arguments, outputs and status word are as for dropkv_score. */
DROPKV_API dropkv_status dropkv_score_noalloc(const dropkv_shape* shape, const void* q_window, const void* k,
                                              const void* v, const int32_t* lengths, int32_t pool_kernel,
                                              int32_t protect, float* scores, float* raw_scores, uint32_t* status,
                                              cudaStream_t stream);

/* Step S5: evict the evict_k[b] lowest scores of every KV head (equal scores:
 * the lower position is evicted first) and list the kept positions.
 *   scores    device float [B][Hkv][n_max] (as written by dropkv_score)
 *   lengths   device int32 [B] or NULL (n_max)
 *   evict_k   device int32 [B]: 0 <= k_b <= n_b - protect (else FLAG_BAD_K, nothing evicted)
 *   protect   the protect value the scores were made with (bounds k_b)
 *   kept_idx  device int32 [B][Hkv][n_max]: first n_b - k_b entries of each
 *             head = kept positions in ascending order; the rest untouched
 *   kept_len  device int32 [B]: n_b - k_b
 * Source: "... output-perturbation scoring", Algorithm 1 summary (evict the
 * smallest scores); "DropKV: Decoupling ...", section 3.2 (bottom-k). */
DROPKV_API dropkv_status dropkv_select(const dropkv_shape* shape, const float* scores, const int32_t* lengths,
                            const int32_t* evict_k, int32_t protect, int32_t* kept_idx, int32_t* kept_len,
                            void* workspace, size_t workspace_bytes, uint32_t* status, cudaStream_t stream);

/* Step S6: gather the kept rows of K and V.
 *   k, v      device bf16 [B][Hkv][n_max][d]
 *   kept_idx, kept_len  as written by dropkv_select
 *   out_rows  row capacity of the outputs per head (>= max_b kept_len[b],
 *             else FLAG_OVERFLOW and only out_rows rows are copied)
 *   k_out, v_out  device bf16 [B][Hkv][out_rows][d], must not overlap k or v;
 *             rows >= kept_len[b] are untouched
 * Source: "DropKV: Decoupling ...", section 2.2 (eviction removes tokens and
 * shrinks the resident cache). */
DROPKV_API dropkv_status dropkv_compact(const dropkv_shape* shape, const void* k, const void* v, const int32_t* kept_idx,
                             const int32_t* kept_len, int32_t out_rows, void* k_out, void* v_out,
                             uint32_t* status, cudaStream_t stream);

/* Step S5 with one pool per sequence (the adaptive head budget of AdaDropKV,
 * "DropKV: Decoupling ...", section 5.3 and Appendix A.3; the pages give no
 * allocation rule, so the plainest is taken): the scores of all KV heads of
 * sequence b compete, and the evict_total[b] smallest (score, head, position)
 * triples are evicted (equal scores: the lower head, then the lower position,
 * goes first), so each head keeps its own number of slots.
 *   scores    device float [B][Hkv][n_max] (as written by dropkv_score)
 *   lengths   device int32 [B] or NULL (n_max)
 *   evict_total  device int32 [B]: 0 <= e_b <= Hkv (n_b - protect) (else
 *             FLAG_BAD_K and nothing evicted); Hkv * k_b gives the same total
 *             budget as dropkv_select
 *   kept_idx  device int32 [B][Hkv][n_max]: first kept_len[b][h] entries of
 *             each head = kept positions ascending; the rest untouched
 *   kept_len  device int32 [B][Hkv]
 * Requires Hkv * n_max < 2^31. */
DROPKV_API dropkv_status dropkv_select_layer(const dropkv_shape* shape, const float* scores, const int32_t* lengths,
                                             const int32_t* evict_total, int32_t protect, int32_t* kept_idx,
                                             int32_t* kept_len, void* workspace, size_t workspace_bytes,
                                             uint32_t* status, cudaStream_t stream);

/* dropkv_compact with a kept count per KV head: kept_len is [B][Hkv] (as
 * written by dropkv_select_layer); everything else as dropkv_compact. */
DROPKV_API dropkv_status dropkv_compact_heads(const dropkv_shape* shape, const void* k, const void* v,
                                              const int32_t* kept_idx, const int32_t* kept_len, int32_t out_rows,
                                              void* k_out, void* v_out, uint32_t* status, cudaStream_t stream);

/* Steps S1-S6 in one call: dropkv_score, dropkv_select and (when k_out and
 * v_out are given) dropkv_compact, with the same arguments, outputs and
 * results as those three calls in sequence.  Every argument is checked before
 * anything is launched.  Heads of at most 8 * 16384 slots have MaxPool1D and
 * protection done inside the selection kernel (the pooled scores are still
 * written to `scores`), one launch fewer than the separate calls.
 *   k_out, v_out  both NULL (no compaction; out_rows ignored) or both set
 * Sources: as for the three calls. */
DROPKV_API dropkv_status dropkv_evict(const dropkv_shape* shape, const void* q_window, const void* k, const void* v,
                                      const int32_t* lengths, const int32_t* evict_k, int32_t pool_kernel,
                                      int32_t protect, float* scores, float* raw_scores, int32_t* kept_idx,
                                      int32_t* kept_len, int32_t out_rows, void* k_out, void* v_out, void* workspace,
                                      size_t workspace_bytes, uint32_t* status, cudaStream_t stream);

/* dropkv_score and dropkv_evict with a score kind (DROPKV_SCORE_DROPKV or
 * DROPKV_SCORE_SNAPKV; anything else is DROPKV_ERR_INVALID_ARG).  With
 * DROPKV_SCORE_SNAPKV the singular rule does not apply (nothing is divided by
 * 1 - p_j), V is read only by the compaction, and the workspace exports lse
 * but not a.  Everything else is as for the calls without the kind. */
DROPKV_API dropkv_status dropkv_score_ex(const dropkv_shape* shape, int32_t score_kind, const void* q_window,
                                         const void* k, const void* v, const int32_t* lengths, int32_t pool_kernel,
                                         int32_t protect, float* scores, float* raw_scores, void* workspace,
                                         size_t workspace_bytes, uint32_t* status, cudaStream_t stream);
DROPKV_API dropkv_status dropkv_evict_ex(const dropkv_shape* shape, int32_t score_kind, const void* q_window,
                                         const void* k, const void* v, const int32_t* lengths, const int32_t* evict_k,
                                         int32_t pool_kernel, int32_t protect, float* scores, float* raw_scores,
                                         int32_t* kept_idx, int32_t* kept_len, int32_t out_rows, void* k_out,
                                         void* v_out, void* workspace, size_t workspace_bytes, uint32_t* status,
                                         cudaStream_t stream);

/* Infrastructure (no passage of the pages): error reporting.
 * Synchronise `stream`, read the device status word and map it to a status
 * (the first of SINGULAR, NONFINITE, DEVICE_ARG, TIMEOUT that is set, else OK;
 * FLAG_INTERNAL maps to DROPKV_ERR_CUDA).
 * *flags_out (if not NULL) receives the raw word. */
DROPKV_API dropkv_status dropkv_read_status(const uint32_t* status, cudaStream_t stream, uint32_t* flags_out);

/* Version string of the library build. */
DROPKV_API const char* dropkv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DROPKV_H */
