/*
 * Token sampling from rows of logits (libattn.so; C ABI).
 *
 * Concept chapter "Forward Pass and Generation", section 3.2: greedy
 * decoding takes the most probable token; temperature T divides the logits
 * before the softmax (section 3.2.2); top-k keeps the k most probable tokens
 * and top-p the smallest set whose probability reaches p (section 3.2.3);
 * the kept tokens are renormalised and sampled.  The code walkthrough's
 * section 4.3: a greedy batch takes the argmax, the others go through
 * temperature and top-k/top-p.
 *
 * Readings where the pages leave a step open:
 *   - ties: greedy returns the smallest index holding the largest logit; the
 *     top-k and top-p limits keep every token whose logit equals the last
 *     kept one;
 *   - top-k and top-p both apply to softmax(logits / T) and the kept set is
 *     their intersection;
 *   - sampling walks the kept tokens in vocabulary order: the token is the
 *     smallest kept index whose cumulative kept probability exceeds
 *     uniform[b] * (kept probability).  The random number is an input.
 */
#ifndef GB300_SAMPLE_H
#define GB300_SAMPLE_H

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One token per row of logits.
 *   logits:      fp32 [B, ld] on the device, row b's V logits first; finite
 *                or -inf, at least one finite value per row.
 *   temperature: fp32 [B] on the device; <= 0 means greedy for that row.
 *   top_k:       int32 [B]; <= 0 or >= V means no top-k limit.
 *   top_p:       fp32 [B]; >= 1 means no top-p limit, <= 0 keeps only the
 *                largest logit (and its ties).
 *   uniform:     fp32 [B], each in [0, 1): the row's random number.
 *   tokens:      int32 [B] on the device (output).
 * All device pointers, caller-owned; asynchronous on `stream`.  Returns
 * ATTN_OK, ATTN_EINVAL (NULL pointer, B < 0, V < 1, V > 2^23, ld < V),
 * ATTN_EDEVICE or ATTN_ELAUNCH.  (Weights are summed exactly as 64-bit
 * integers in units of 2^-40, which bounds V by 2^23.) */
ATTN_API int attn_sample_tokens(const float* logits, int32_t B, int32_t V, int64_t ld,
                                const float* temperature, const int32_t* top_k, const float* top_p,
                                const float* uniform, int32_t* tokens, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_SAMPLE_H */
