/*
 * tf_paged_mla.h -- attention over a paged latent (MLA) KV cache on one GB300.
 *
 * The problem, as the TensorFold pages state it:
 *  - each token's cache row is 512 bf16 latent values plus a 64-value bf16 rope
 *    key (issue #1142, "What happens now": 12 caches x (1,024 + 64) bytes; 64 bytes
 *    cannot hold 64 bf16 values, so the rope key is stored as 64 bf16 and a row of
 *    one cache is 1,152 B);
 *  - rows sit in 512-row pages taken from one shared pool; a stream maps its
 *    logical pages to pool pages through a page table, and the cache kernels take
 *    that table plus the elements between pages (issue #1142, "GLM declares a
 *    kv_pool.Layout"); a null table keeps contiguous rows: a window is its pages taken in
 *    order, under the same addressing rule (issue #1313, step 1.3);
 *  - taken pages can be filled with NaN so that a read before a write shows
 *    (issue #1142, same section: TF_KV_POISON=1);
 *  - streams share prefix pages by reference the way the radix prompt store keeps
 *    them (PR #1732, "What this changes");
 *  - a kept state copies only its first `at` rows (issue #1142, piece 1);
 *  - every head's absorbed query is read against the one latent (issue #1313,
 *    step 2, decode bullet), over 1-2 causal query rows for MTP drafts (PR #1732,
 *    lookahead of 1) or a T-row prefill chunk against its prefix (chunked-prefill
 *    note, section 1).
 *
 * Conventions for every call:
 *  - Return 0 (TF_OK) or a negative TF_E_* code.  Arguments are checked on the
 *    host before anything is launched; a failed check launches nothing.
 *  - Pointers named d_* are device pointers, h_* host pointers.  All device
 *    memory (the pool, page tables, queries, outputs, workspace) belongs to the
 *    caller; the library never allocates or frees device memory.  tf_kvpool
 *    objects are host memory owned by the library until tf_kvpool_destroy.
 *  - Launches are asynchronous on the given CUDA stream (cudaStream_t passed as
 *    void*; NULL is the legacy default stream).  No call synchronises except
 *    tf_last_error and tf_profile_read.
 *  - Errors found by a kernel (a page id outside the pool, a bounded wait that
 *    ran out) are recorded in a device error word inside the pool's memory; the
 *    kernel skips the bad access and never traps.  tf_last_error reads them.
 *  - bf16 is passed as raw 16-bit patterns.
 */
#ifndef TF_PAGED_MLA_H
#define TF_PAGED_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TF_OK 0
#define TF_E_ARG (-1)          /* a null pointer, a bad size or a bad flag */
#define TF_E_RANGE (-2)        /* an id, length or position outside what the pool holds */
#define TF_E_NOMEM (-3)        /* the pool has too few free pages, or a buffer is too small */
#define TF_E_CUDA (-4)         /* a CUDA runtime or driver call failed */
#define TF_E_TIMEOUT (-5)      /* a kernel's bounded wait ran out (device error word) */
#define TF_E_UNSUPPORTED (-6)  /* a shape this library does not handle */
#define TF_E_DEVICE (-7)       /* a kernel met a bad page id (device error word) */

#define TF_PAGE_ROWS 512
#define TF_LATENT_DIM 512
#define TF_ROPE_DIM 64
#define TF_QK_DIM 576
#define TF_MAX_STREAMS 512
#define TF_MAX_HEADS 128
#define TF_POOL_POISON 1u      /* fill pages with bf16 NaN (0x7FC0) when they are taken */
#define TF_POOL_BATCH_INVARIANT 2u  /* attention on this pool: a stream's result has the same
                                       bits whatever else is in the batch (see tf_paged_mla_attend) */
#define TF_POOL_FP8 4u              /* FP8 latent rows (see "FP8 pages" below) */

/* ---- FP8 pages (issue #1313, step 1.3, item 3: FP8 latent rows on pages, a page's fp32 row
 * scales stored behind its rows; windows laid out the same way) ----
 * With TF_POOL_FP8 a page of one cache is
 *   latent codes  512 rows x 512 bytes, OCP FP8 E4M3 (bias 7, largest finite 448)   262,144 B
 *   scales        512 fp32, one a row                                                  2,048 B
 *   rope          512 rows x 64 bf16, as on BF16 pages                                65,536 B
 * = 329,728 bytes (644 a row and cache instead of 1,152).  Row r's latent value i is
 * code_r[i] * scale_r.  tf_paged_append takes the same bf16 rows as on a BF16 pool and
 * quantizes each latent row: amax = max_i |x_i|, scale = amax / 448 (fp32 division), code_i =
 * E4M3(x_i / scale) rounded to nearest even with saturation to +-448 (fp32 division); a row of
 * zeros stores scale 0 and codes 0.  Inputs must be finite.  tf_paged_mla_attend computes the
 * same attention over the dequantized rows, each value taken as bf16(code * scale): the kernel
 * reads the codes and expands each key tile in shared memory (the workspace is as on a BF16
 * pool); on a TF_POOL_BATCH_INVARIANT pool the rows are first expanded to bf16 pages in the
 * workspace, whose size then includes them.  tf_state_copy_rows copies codes, scales and rope
 * of rows [0, at).  Poison fills taken pages with 0xFF bytes (NaN in all three blocks).
 * tf_paged_mla_attend_sparse gathers the listed rows' codes and scales and expands them the
 * same way.  tf_paged_mla_attend_static returns TF_E_UNSUPPORTED on a batch-invariant FP8 pool. */

typedef struct tf_kvpool tf_kvpool;

/* A pool of num_pages pages for each of num_caches caches.  One page of one cache
 * is page_rows x latent_dim bf16 (the latent block) followed by page_rows x
 * rope_dim bf16 (the rope block): 589,824 bytes at 512/512/64 (329,728 with
 * TF_POOL_FP8, see "FP8 pages").  Cache c's page p
 * starts at dev_base + (c * num_pages + p) * page_bytes.  A page id names the same
 * page in every cache (a token's rows in all caches live under one id). */
typedef struct {
    int32_t num_caches;  /* 1 .. 65,535 (12 for 11 MLA layers plus the MTP layer) */
    int32_t num_pages;   /* >= 1; num_caches * num_pages < 2^31 */
    int32_t page_rows;   /* must be 512 */
    int32_t latent_dim;  /* must be 512 */
    int32_t rope_dim;    /* must be 64 */
    uint32_t flags;      /* TF_POOL_POISON | TF_POOL_BATCH_INVARIANT | TF_POOL_FP8, or 0 */
    uint64_t seed;       /* 0: free pages are handed out in id order; else in a seeded permutation */
} tf_kvpool_desc;

/* Device bytes a pool with this descriptor needs: every page of every cache plus
 * a 256-byte control block (the device error word) after the last page.
 * Returns 0 for an invalid descriptor. */
size_t tf_kvpool_bytes(const tf_kvpool_desc *desc);

/* Make a pool over caller memory dev_base (>= tf_kvpool_bytes, 1024-byte aligned).
 * All pages start free with refcount 0.  Touches no device memory: the device
 * error word is zeroed, asynchronously, on the stream of the pool's first launch.
 * On success *out owns host state only; the device memory stays the caller's.
 * TF_E_ARG for a null pointer, an invalid descriptor or an unaligned dev_base;
 * TF_E_NOMEM if dev_bytes < tf_kvpool_bytes(desc). */
int tf_kvpool_create(const tf_kvpool_desc *desc, void *dev_base, size_t dev_bytes, tf_kvpool **out);

/* Free the host state.  The device memory is untouched.  TF_E_ARG for NULL. */
int tf_kvpool_destroy(tf_kvpool *pool);

/* Take n free pages (refcount 1) into h_ids_out[n].  With TF_POOL_POISON the taken
 * pages of every cache are NaN-filled on cuda_stream before the call returns
 * (asynchronously).  TF_E_NOMEM, and nothing taken, if fewer than n are free;
 * TF_E_ARG for n < 0 or a null h_ids_out with n > 0. */
int tf_kvpool_take(tf_kvpool *pool, int32_t n, int32_t *h_ids_out, void *cuda_stream);

/* Add one reference to each of n taken pages: a kept state or a second stream
 * holding a prefix page (PR #1732: kept states hold prefix pages by reference).
 * TF_E_RANGE, and nothing changed, if any id is not taken; TF_E_ARG as for take. */
int tf_kvpool_ref(tf_kvpool *pool, const int32_t *h_ids, int32_t n);

/* Drop one reference from each of n pages; a page whose count reaches 0 is free
 * again.  TF_E_RANGE, and nothing changed, if any id is not taken (an id listed
 * k times must hold k references); TF_E_ARG as for take. */
int tf_kvpool_release(tf_kvpool *pool, const int32_t *h_ids, int32_t n);

/* Free pages now, and one page's reference count (-1 for a bad id). */
int32_t tf_kvpool_free_pages(const tf_kvpool *pool);
int32_t tf_kvpool_refcount(const tf_kvpool *pool, int32_t id);

/* Device address of cache c's page p (NULL for bad arguments). */
void *tf_kvpool_page_ptr(const tf_kvpool *pool, int32_t cache, int32_t page);

/* ---- the kv_pool plan (issue #1313, "Why" bullet 3 and "Proposal" step 1.1) ----
 * Host arithmetic only.  Order: one window of pages for the engine's own sequence
 * (ceil((context + lookahead) / page_rows) pages), then either a page for each
 * other stream (today's order) or, with engine_paged, as many windows as the room
 * holds, n = min(lanes, 1 + (room - window) / (window + fixed)), at least one,
 * the streams holding max(n windows, one window + lanes - 1 pages); then each
 * other stream's fixed bytes; then the prompt cache up to its budget; then the
 * remaining room as more pages.  TF_E_NOMEM if the room cannot hold the streams;
 * TF_E_ARG for a null pointer, a negative byte count, budget or lookahead, or a
 * context, lanes, page_rows or bytes_per_token below 1. */
typedef struct {
    int64_t room_bytes;
    int64_t context_tokens;
    int32_t lanes;              /* --parallel */
    int32_t page_rows;          /* 512 */
    int32_t lookahead;          /* MTP lookahead rows, 1 */
    int32_t engine_paged;       /* 0: today's order; 1: step 1 */
    int64_t bytes_per_token;    /* all caches of one token, e.g. 13,056 */
    int64_t fixed_bytes;        /* fixed state of each other stream */
    int64_t cache_budget_bytes; /* prompt cache budget */
} tf_plan_in;

typedef struct {
    int32_t n_windows;
    int64_t window_pages;
    int64_t stream_pages;
    int64_t cache_bytes;
    int64_t other_pages;
    int64_t pool_pages;
    int64_t pool_tokens;
} tf_plan_out;

int tf_kvpool_plan(const tf_plan_in *in, tf_plan_out *out);

/* ---- paged append (issue #1142: the row-writing kernel takes the page table) ----
 * For every stream s < S and new row i < n, row pos = h_pos[s] + i is written to
 * pool page pt[s][pos / 512], row pos % 512, of cache `cache`: 512 latent values
 * from d_latent[s][i][:] and 64 rope values from d_rope[s][i][:] (bf16).
 * d_pt: int32 [S][max_pages] device table, or NULL for contiguous windows
 * (stream s's logical page j is pool page s * max_pages + j).
 * h_pos: host int64 [S]; every pos + n must be <= max_pages * 512.
 * d_latent and d_rope must be 16-byte aligned.
 * A table entry outside [0, num_pages) is recorded as TF_E_DEVICE and that row
 * is skipped.  Bit-exact: the bytes are copied, never converted (FP8 pools quantize).
 * Errors: TF_E_ARG for a null pool or h_pos, S outside [1, TF_MAX_STREAMS], n < 0,
 * max_pages < 1, null or unaligned row buffers with n > 0; TF_E_RANGE for a cache
 * outside the pool, a position outside the table, or a NULL table wider than the
 * pool (S * max_pages > num_pages).  n == 0 launches nothing. */
int tf_paged_append(tf_kvpool *pool, int32_t cache, const int32_t *d_pt, int32_t max_pages,
                    const int64_t *h_pos, int32_t S, int32_t n,
                    const void *d_latent, const void *d_rope, void *cuda_stream);

/* ---- attention over the pages (issue #1313 step 2 decode bullet; issue #1142
 * "What stays as it is": the same 512-key chunks merged in the same order) ----
 * For stream s, query row r (position p = h_len[s] - R + r) and head h:
 *   s_j = scale * (q[s][r][h][0:512] . C_j + q[s][r][h][512:576] . Kr_j), j = 0..p
 *   out[s][r][h][:] = sum_j softmax(s)_j * C_j      (bf16, 512 values)
 *   lse[s][r][h]    = log sum_j exp(s_j)           (fp32, natural log; d_lse may be NULL)
 * where C_j / Kr_j are the latent / rope parts of the stream's row j, read
 * through d_pt (or contiguous windows when d_pt is NULL, as in tf_paged_append).
 * R = 1-2 is decode (MTP drafts); R > 2 is a prefill chunk.  h_len: host int64
 * [S], rows after the current rows were appended, each >= R and <= max_pages * 512.
 * d_q: bf16 [S][R][H][576]; d_out: bf16 [S][R][H][512]; d_lse: fp32 [S][R][H].
 * How the keys are shared out decides the order of the fp32 sums, never which keys
 * count; a stream's result never depends on which pool pages hold its rows.
 *  - Default: the key tiles of the batch are cut into near-equal contiguous ranges,
 *    one a CTA (decode, MTP rows), or the (stream, row group) units of a prefill
 *    chunk, each read only to the last key its rows see, are numbered tile by tile
 *    and cut the same way.  Every SM gets the same work whatever the mix of lengths;
 *    a stream's bits may differ (within rounding) between batches, and are identical
 *    between calls on the same batch.
 *  - Pools made with TF_POOL_BATCH_INVARIANT: each stream's keys are cut into splits
 *    whose bounds depend on that stream's length alone and merged in split order,
 *    as the pages' engine does with its fixed key chunks, so a stream attended in a
 *    batch equals the same stream attended alone, bit for bit.
 * d_ws: caller workspace of at least tf_paged_mla_workspace_bytes(pool, ...) bytes,
 * 256-byte aligned, used for the split partials (fp32); it may be NULL only when
 * that size is 0.  Rows past h_len[s] are never read into the result (they may
 * hold NaN).  Limits: 1 <= S <= TF_MAX_STREAMS, 1 <= H <= TF_MAX_HEADS, scale a
 * finite number > 0, d_q and d_out 16-byte aligned (TF_E_ARG otherwise); h_len[s] <=
 * INT32_MAX (TF_E_UNSUPPORTED otherwise, and a workspace size of 0).  TF_E_RANGE for a
 * cache outside the pool, a length below R or past the table, or a NULL table wider than
 * the pool; TF_E_NOMEM for a workspace smaller than needed (TF_E_ARG if it is NULL or
 * not 256-byte aligned). */
size_t tf_paged_mla_workspace_bytes(const tf_kvpool *pool, int32_t S, int32_t R, int32_t H,
                                    const int64_t *h_len);   /* pool may be NULL: default plan */

int tf_paged_mla_attend(tf_kvpool *pool, int32_t cache, const int32_t *d_pt, int32_t max_pages,
                        const int64_t *h_len, int32_t S, int32_t R, int32_t H,
                        const void *d_q, float scale, void *d_out, float *d_lse,
                        void *d_ws, size_t ws_bytes, void *cuda_stream);

/* ---- attention without a caller workspace ----
 * No counterpart on the TensorFold pages: this entry point exists for callers of
 * this library that cannot allocate device memory -- an engine that hands the
 * library only its page pool and per-step tensors from a fixed arena and allows no
 * further device allocation while it serves, or a host program that has no device
 * allocator of its own.  It computes exactly what tf_paged_mla_attend computes, with
 * the same arguments minus the workspace: the split partials go to one scratch
 * array of TF_STATIC_WS_BYTES (64 MiB) that the library defines in device memory.
 * Every GPU that loads the library holds that array until the process exits.
 * - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * - The first call on each device looks up the array's device address with that
 *   device current (cudaGetSymbolAddress) and remembers it; make that first call
 *   before any stream capture.
 * - On a default pool the partials are bounded by the launch's CTA ranges (two
 *   slots of 128 KiB a CTA, at most 240 CTAs), so every valid call fits.  On a
 *   TF_POOL_BATCH_INVARIANT pool they grow with the lengths; a call that would need
 *   more than TF_STATIC_WS_BYTES (see tf_paged_mla_workspace_bytes) returns
 *   TF_E_NOMEM and launches nothing.
 * - Every call shares the one array and it keeps the last call's contents (each
 *   call writes every partial it reads, so nothing has to start at zero).  Calls
 *   that overlap on the GPU -- on two streams, or from two threads -- race on it:
 *   order them on one stream, or use tf_paged_mla_attend with separate workspaces. */
#define TF_STATIC_WS_BYTES (64u << 20)

/* ---- attention over listed rows (issue #1313, step 2: a sparse decode row touches at most
 * 2,048 latent rows; issue #1142, section 2: both the dense
 * latent kernels and the sparse gather are given the page table; "What stays as it is": the sparse path reads the same rows) ----
 * One query row a stream (R = 1).  Stream s's keys are the rows d_idx[s][0 .. h_nidx[s]) of the
 * stream (row numbers as in tf_paged_mla_attend, each < h_len[s]), in list order:
 *   s_j = scale * (q[s][h][0:512] . C_idx[j] + q[s][h][512:576] . Kr_idx[j])
 *   out[s][h][:] = sum_j softmax(s)_j * C_idx[j];  lse[s][h] = log sum_j exp(s_j).
 * A row listed twice counts twice.  d_idx: int32 [S][max_idx] device; entries past h_nidx[s] are
 * not read.  d_q: bf16 [S][H][576]; d_out: bf16 [S][H][512]; d_lse: fp32 [S][H] or NULL.
 * Each row is fetched through d_pt (or the contiguous windows of a NULL table) with TMA gathers.
 * A listed row outside [0, h_len[s]) or a table entry outside the pool is recorded as
 * TF_E_DEVICE and the call's output is undefined.  Limits: 1 <= h_nidx[s] <= max_idx (TF_E_RANGE
 * otherwise), S, H, scale, alignment, lengths and workspace as for tf_paged_mla_attend; h_len[s] <= INT32_MAX and the pool must have fewer than 2^31 / 4,608
 * pages over all caches (TF_E_UNSUPPORTED otherwise).  The keys are dealt out as in the default plan of tf_paged_mla_attend
 * (whatever the pool's flags); d_ws holds the partials as there. */
size_t tf_paged_mla_sparse_workspace_bytes(const tf_kvpool *pool, int32_t S, int32_t H, const int32_t *h_nidx);

int tf_paged_mla_attend_sparse(tf_kvpool *pool, int32_t cache, const int32_t *d_pt, int32_t max_pages,
                               const int64_t *h_len, const int32_t *d_idx, int32_t max_idx, const int32_t *h_nidx,
                               int32_t S, int32_t H, const void *d_q, float scale, void *d_out, float *d_lse,
                               void *d_ws, size_t ws_bytes, void *cuda_stream);

int tf_paged_mla_attend_static(tf_kvpool *pool, int32_t cache, const int32_t *d_pt, int32_t max_pages,
                               const int64_t *h_len, int32_t S, int32_t R, int32_t H,
                               const void *d_q, float scale, void *d_out, float *d_lse, void *cuda_stream);

/* ---- kept-state copy (issue #1142, piece 1: keepAs / restoreState copy each
 * cache's first `at` rows; rows past `at` are never read) ----
 * Copies rows [0, at) of cache `cache` (every cache when cache < 0) from the
 * pages d_src_pages[0 .. ceil(at/512)) to the pages d_dst_pages[same], row for
 * row.  Rows at and past `at` of the last page are neither read nor written.
 * Page ids outside the pool are recorded as TF_E_DEVICE and skipped.  Bit-exact.
 * TF_E_ARG for a null pool, at < 0, or null tables with at > 0; TF_E_RANGE for a
 * cache >= num_caches or at > num_pages * 512.  at == 0 launches nothing. */
int tf_state_copy_rows(tf_kvpool *pool, int32_t cache, const int32_t *d_src_pages,
                       const int32_t *d_dst_pages, int64_t at, void *cuda_stream);

/* ---- diagnostics (not on the hot path) ---- */

/* Synchronise the device, read and clear the pool's device error word.
 * Returns TF_OK, TF_E_DEVICE or TF_E_TIMEOUT; *detail (may be NULL) gets the
 * offending value (a page id or a wait site). */
int tf_last_error(tf_kvpool *pool, int64_t *detail);

/* Check that a bounded device wait really ends: launch a one-block kernel that
 * waits on a barrier nothing completes, with a limit of limit_cycles SM clock
 * cycles (1 .. 2^32), the same wait every kernel here uses.  The wait gives up,
 * records TF_E_TIMEOUT (detail 99) in the pool's error word and the kernel returns;
 * read it with tf_last_error.  No counterpart on the pages: it exercises this
 * library's own failure path without faulting or hanging the GPU. */
int tf_diag_wait_timeout(tf_kvpool *pool, int64_t limit_cycles, void *cuda_stream);

/* The work plan tf_paged_mla_attend would use for these lengths, for inspection: host
 * arithmetic only, nothing launched.  sms: the SMs to plan for (<= 0: the current device's,
 * or TF_PLAN_MAX_RANGES without one); invariant != 0: a TF_POOL_BATCH_INVARIANT pool.
 *   info->mode     0 key-tile ranges (decode, MTP rows), 1 key-tile ranges over (stream,
 *                  column group) units, one CTA a range (prefill chunks), 2 per-stream splits
 *                  (batch-invariant pools)
 *   info->ctas     CTAs launched
 *   info->nranges  mode 0: ranges (each taken by info->groups CTAs side by side); mode 1:
 *                  ranges (= ctas); else 0
 *   info->groups   column groups a stream: ceil(R * H / 64)
 *   info->work     mode 0: 64-key tiles of the batch; mode 1: units; mode 2: (split, group) items
 *   info->slots    fp32 partial slots in the workspace (0: no combine pass)
 * range_bounds (may be NULL): the nranges + 1 bounds of the ranges (at most TF_PLAN_MAX_RANGES
 * + 1 entries).  Mode 0: tile numbers, tiles numbered stream by stream.  Mode 1: positions
 * unit * 2^32 + tile, units numbered stream-major (unit = s * groups + g), each unit as many
 * 64-key tiles as its last column sees (len - R + 1 + that column's row).
 * split_keys (may be NULL): with mode 2, the keys of one split of each stream [S].
 * TF_E_ARG for a null h_len or info, or S, R, H outside the attention's limits; TF_E_UNSUPPORTED
 * for S * R * H above 2^30 (as tf_paged_mla_attend); TF_E_RANGE for a length below R or above
 * INT32_MAX. */
#define TF_PLAN_MAX_RANGES 240
typedef struct {
    int32_t mode, ctas, nranges, groups;
    int64_t work, slots;
} tf_attend_plan;
int tf_paged_mla_plan_info(int32_t S, int32_t R, int32_t H, const int64_t *h_len, int32_t sms, int32_t invariant,
                           tf_attend_plan *info, int64_t *range_bounds, int64_t *split_keys);

/* Kernels this library has launched since the process started. */
int64_t tf_launch_count(void);

/* With on != 0, every launch made for this pool is bracketed by CUDA events on
 * its stream.  tf_profile_read synchronises on them and returns, for kernel
 * kind `kind` (0 append, 1 attention main pass, 2 split combine, 3 state copy,
 * 4 poison fill), the summed milliseconds and the launch count since the last
 * read, then forgets them. */
int tf_profile_enable(tf_kvpool *pool, int32_t on);
int tf_profile_read(tf_kvpool *pool, int32_t kind, double *total_ms, int64_t *launches);

#ifdef __cplusplus
}
#endif
#endif /* TF_PAGED_MLA_H */
