/*
 * Blocked top-k with an exact merge, for the logits an indexer writes before sparse attention.
 *
 * Source: "Running CHUNKED_PREFILL_SIZE above 1024 without the long-prompt memory problem",
 * section 2.3 (block the indexer along the key axis and merge top-k).  Each block of keys keeps
 * its own top-k (values and indices); the top-k of the concatenated candidates is the top-k of
 * the whole row.  The identity is exact, so the blocked result equals the unblocked one.  The
 * selected indices are what tf_paged_mla_attend_sparse takes as its listed rows.
 *
 * Order.  A row's keys are ranked by value, larger first, under the IEEE total order of fp32:
 * -0 ranks below +0 and a NaN ranks below every number (-inf included).  Equal values rank by
 * their column, smaller first.  Under this order every row has exactly one top-k, so the result
 * is bit-exact and does not depend on the block size or on the order in which blocks finish.
 *
 * Conventions as in tf_paged_mla.h: device pointers are prefixed d_, calls are asynchronous on
 * `stream` (a cudaStream_t, 0 for the legacy stream), TF_OK or a negative TF_E_* code.
 */
#ifndef TF_TOPK_H
#define TF_TOPK_H

#include <stddef.h>
#include <stdint.h>

#include "tf_paged_mla.h"

#ifdef __cplusplus
extern "C" {
#endif

#define TF_TOPK_MAX_K 2048
#define TF_TOPK_BLOCK 16384 /* keys a first-level block holds (one CTA each) */
#define TF_TOPK_MERGE 8192  /* candidates a merge block holds */

/* Device workspace for tf_topk_blocked: the candidates of every level but the last,
 * 8 bytes each (a key and a column).  Zero when every row fits one block. */
size_t tf_topk_workspace_bytes(int64_t rows, int64_t n, int32_t k);

/* Top-k of each row of a row-major fp32 matrix, sorted best first.
 *
 * d_logits: [rows][ld] fp32, row r's keys in columns [0, len_r); 16-byte aligned, ld a
 *   multiple of 4 and ld >= n.  The caller owns it; it is only read.
 * d_len: [rows] int32 row lengths (NULL: every row has n keys); each is clamped to [0, n].
 * k: 1 <= k <= TF_TOPK_MAX_K.
 * d_idx: [rows][k] int32 out, the columns of the k best keys, best first.
 * d_val: [rows][k] fp32 out, their values, copied bit for bit from d_logits.
 *   A row with fewer than k keys fills its tail with column -1 and value -inf.
 * d_ws / ws_bytes: device workspace of at least tf_topk_workspace_bytes(rows, n, k) bytes,
 *   16-byte aligned (may be NULL when that is zero).
 *
 * The first level cuts each row into blocks of TF_TOPK_BLOCK keys and keeps every block's
 * top-k; each later level cuts the candidates into blocks of TF_TOPK_MERGE and keeps their
 * top-k, until one block is left, whose top-k is sorted and written.  One kernel launch a
 * level; the levels are ordered on `stream`.
 *
 * Errors: TF_E_ARG for a null pointer, rows < 0, n < 0, ld < n, an unaligned d_logits or ld,
 * or k outside [1, TF_TOPK_MAX_K]; TF_E_UNSUPPORTED for n > INT32_MAX, rows > INT32_MAX or more
 * than INT32_MAX blocks in a level; TF_E_NOMEM if ws_bytes is too small; TF_E_CUDA if a launch
 * fails.  rows == 0 (with valid sizes) launches nothing and may pass NULL pointers. */
int tf_topk_blocked(const float *d_logits, int64_t rows, int64_t n, int64_t ld, const int32_t *d_len, int32_t k,
                    int32_t *d_idx, float *d_val, void *d_ws, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TF_TOPK_H */
