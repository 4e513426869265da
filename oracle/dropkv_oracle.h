/*
 * DropKV scoring path: CPU oracle (fp64).  TEST INFRASTRUCTURE ONLY: used by
 * the test suite, the smoke check and the benchmark's CPU-baseline leg, never
 * by the product library.  See dropkv_oracle.c for the definitions and their
 * sources.
 */
#ifndef DROPKV_ORACLE_H
#define DROPKV_ORACLE_H
#include <stdint.h>

typedef struct { int32_t B, Hq, Hkv, d, n_max, w; } oracle_shape;

enum { ORACLE_OK = 0, ORACLE_INVALID = 1, ORACLE_SINGULAR = 3, ORACLE_NOMEM = 9 };
enum { ORACLE_F64 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_KIND_DROPKV = 0, ORACLE_KIND_SNAPKV = 1 };

/* Window attention + scores.  q [B,Hq,w,d], k/v [B,Hkv,n_max,d] (fp64 values or
 * bf16 bit patterns, per dtype).  m/l [B,Hq,w], a [B,Hq,w,d] (nullable),
 * raw/final [B,Hkv,n_max]; slots j >= n_b are set to NaN.  Returns
 * ORACLE_SINGULAR (and the unit b*Hkv+h) if some p_j equals 1. */
int oracle_score(const oracle_shape* s, int dtype, const void* q, const void* k, const void* v,
                 const int32_t* lengths, int pool_kernel, int protect,
                 double* m_out, double* l_out, double* a_out, double* raw_out, double* final_out,
                 int nthreads, int32_t* singular_unit);

/* oracle_score with a score kind: ORACLE_KIND_DROPKV (the perturbation score,
 * as oracle_score) or ORACLE_KIND_SNAPKV (window sum of p_j, no singular rule). */
int oracle_score_kind(const oracle_shape* s, int kind, int dtype, const void* q, const void* k, const void* v,
                      const int32_t* lengths, int pool_kernel, int protect,
                      double* m_out, double* l_out, double* a_out, double* raw_out, double* final_out,
                      int nthreads, int32_t* singular_unit);

/* Bottom-k eviction: kept_idx [B,Hkv,n_max] (first kept_len[b] entries, ascending). */
int oracle_select(const oracle_shape* s, const double* final_scores, const int32_t* lengths,
                  const int32_t* evict_k, int protect, int32_t* kept_idx, int32_t* kept_len);

/* Layer-wide bottom-k: per sequence, evict the evict_total[b] smallest
 * (score, head, position) over all KV heads; kept_len [B,Hkv]. */
int oracle_select_layer(const oracle_shape* s, const double* final_scores, const int32_t* lengths,
                        const int32_t* evict_total, int protect, int32_t* kept_idx, int32_t* kept_len);

/* Gather with a kept count per KV head (kept_len [B,Hkv]). */
int oracle_compact_heads(const oracle_shape* s, int elem_bytes, const void* k, const void* v,
                         const int32_t* kept_idx, const int32_t* kept_len, int out_rows,
                         void* k_out, void* v_out);

/* Gather of kept rows: k_out/v_out [B,Hkv,out_rows,d] of elem_bytes elements. */
int oracle_compact(const oracle_shape* s, int elem_bytes, const void* k, const void* v,
                   const int32_t* kept_idx, const int32_t* kept_len, int out_rows,
                   void* k_out, void* v_out);
/* Causal prefill attention: out[b][hq][i] = sum_{j <= i} p_j v_j for every
 * row i < n_b (rows >= n_b set to NaN).  q [B,Hq,n_max,d], k/v [B,Hkv,n_max,d],
 * out [B,Hq,n_max,d]; s->w is not used. */
int oracle_prefill_attention(const oracle_shape* s, int dtype, const void* q, const void* k, const void* v,
                             const int32_t* lengths, double* out, int nthreads);
#endif
