/* Test hooks of libdropkv, exported ONLY by the test build
 * (libdropkv_test_hooks.so, compiled with -DDROPKV_TEST_HOOKS); the product
 * library libdropkv.so exports none of them.
 *
 * Infrastructure (no passage of the pages): the pipeline failure-detection
 * test drives a real scoring call into its timeout exit without a GPU fault.
 * In the test build every pipeline wait gives up after 10 ms (1 s in the
 * product build).
 */
#ifndef DROPKV_TEST_HOOKS_H
#define DROPKV_TEST_HOOKS_H

#include "dropkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* From the next scoring call on, the scoring pass (pass 2) leaves out the K
 * tile copy of (unit = b * Hkv + h, tile = 128-key tile index): the tile's
 * full-barrier never completes, the MMA issuer's bounded wait runs out, the
 * CTA raises DROPKV_FLAG_TIMEOUT, waits (bounded) for its copies and MMAs in
 * flight, releases its tensor memory and returns; the other CTAs finish
 * normally.  (-1, -1) switches the hook off.  Host-synchronous (a copy to a
 * device symbol); returns DROPKV_ERR_CUDA if that copy fails. */
DROPKV_API dropkv_status dropkv_test_skip_pass2_k(int32_t unit, int32_t tile);

/* The same for the prefill attention (dropkv_evict_prefill,
 * dropkv_prefill_attention): every CTA of (unit, key tile) leaves that K tile
 * copy out, its MMA issuer's wait runs out, and the CTA takes the same exit.
 * (-1, -1) switches the hook off. */
DROPKV_API dropkv_status dropkv_test_skip_prefill_k(int32_t unit, int32_t tile);

#ifdef __cplusplus
}
#endif
#endif /* DROPKV_TEST_HOOKS_H */
