// Host side of the library: the page pool (ids, reference counts, poison on take),
// the kv_pool plan arithmetic, argument checks for every entry point, the device
// error word and launch profiling.  Nothing here touches device memory except the
// error word (zeroed before the first launch, read by tf_last_error) and the
// kernels it launches.
#include <cstdio>
#include <cstring>
#include <new>

#include "tf_internal.h"

namespace tf {

std::atomic<int64_t> &launch_counter() {
    static std::atomic<int64_t> c{0};
    return c;
}

ProfScope::ProfScope(tf_kvpool *p, int k, cudaStream_t s) : pool(p), kind(k), stream(s) {
    if (!pool || !pool->prof) return;
    std::lock_guard<std::mutex> g(pool->mu);
    for (cudaEvent_t *e : {&a, &b}) {
        if (!pool->spare_events.empty()) {
            *e = pool->spare_events.back();
            pool->spare_events.pop_back();
        } else if (cudaEventCreate(e) != cudaSuccess) {
            *e = nullptr;
        }
    }
    if (a) cudaEventRecord(a, stream);
}

ProfScope::~ProfScope() {
    if (!a || !b) return;
    cudaEventRecord(b, stream);
    std::lock_guard<std::mutex> g(pool->mu);
    pool->recs.push_back(ProfRec{kind, a, b});
}

}  // namespace tf

using namespace tf;

static bool desc_ok(const tf_kvpool_desc *d) {
    // the poison and state-copy launches put the caches on the grid's y dimension (at most 65,535)
    return d && d->num_caches >= 1 && d->num_caches <= 65535 && d->num_pages >= 1 && d->page_rows == kPageRows &&
           d->latent_dim == kLat &&
           d->rope_dim == kRope && (d->flags & ~(TF_POOL_POISON | TF_POOL_BATCH_INVARIANT | TF_POOL_FP8)) == 0 &&
           (uint64_t)d->num_caches * (uint64_t)d->num_pages < (1ull << 31);
}

extern "C" size_t tf_kvpool_bytes(const tf_kvpool_desc *d) {
    if (!desc_ok(d)) return 0;
    return (size_t)d->num_caches * (size_t)d->num_pages * page_bytes(*d) + kCtrlBytes;
}

// splitmix64: a published 64-bit mixer, used only to shuffle the free list.
static uint64_t splitmix64(uint64_t &x) {
    uint64_t z = (x += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

extern "C" int tf_kvpool_create(const tf_kvpool_desc *d, void *dev_base, size_t dev_bytes, tf_kvpool **out) {
    if (!out) return TF_E_ARG;
    *out = nullptr;
    if (!desc_ok(d) || !dev_base) return TF_E_ARG;
    if ((reinterpret_cast<uintptr_t>(dev_base) & 1023u) != 0) return TF_E_ARG;
    size_t need = tf_kvpool_bytes(d);
    if (dev_bytes < need) return TF_E_NOMEM;
    tf_kvpool *p = new (std::nothrow) tf_kvpool();
    if (!p) return TF_E_NOMEM;
    p->desc = *d;
    p->base = static_cast<char *>(dev_base);
    p->bytes = dev_bytes;
    p->err = reinterpret_cast<DevErr *>(p->base + need - kCtrlBytes);
    p->refcnt.assign(d->num_pages, 0);
    p->free_ring.resize(d->num_pages);
    for (int i = 0; i < d->num_pages; ++i) p->free_ring[i] = i;
    if (d->seed) {  // Fisher-Yates with a seeded mixer
        uint64_t st = d->seed;
        for (int i = d->num_pages - 1; i > 0; --i) {
            int j = (int)(splitmix64(st) % (uint64_t)(i + 1));
            std::swap(p->free_ring[i], p->free_ring[j]);
        }
    }
    p->free_head = 0;
    p->free_count = d->num_pages;
    *out = p;
    return TF_OK;
}

extern "C" int tf_kvpool_destroy(tf_kvpool *p) {
    if (!p) return TF_E_ARG;
    for (auto &r : p->recs) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    for (auto e : p->spare_events) cudaEventDestroy(e);
    delete p;
    return TF_OK;
}

extern "C" int tf_kvpool_take(tf_kvpool *p, int32_t n, int32_t *ids, void *stream) {
    if (!p || n < 0 || (n > 0 && !ids)) return TF_E_ARG;
    {
        std::lock_guard<std::mutex> g(p->mu);
        if ((size_t)n > p->free_count) return TF_E_NOMEM;
        const size_t N = p->free_ring.size();
        for (int i = 0; i < n; ++i) {
            int32_t id = p->free_ring[(p->free_head + i) % N];
            ids[i] = id;
            p->refcnt[id] = 1;
        }
        p->free_head = (p->free_head + n) % N;
        p->free_count -= n;
    }
    if (n > 0 && (p->desc.flags & TF_POOL_POISON)) return launch_poison(p, ids, n, (cudaStream_t)stream);
    return TF_OK;
}

extern "C" int tf_kvpool_ref(tf_kvpool *p, const int32_t *ids, int32_t n) {
    if (!p || n < 0 || (n > 0 && !ids)) return TF_E_ARG;
    std::lock_guard<std::mutex> g(p->mu);
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= p->desc.num_pages || p->refcnt[ids[i]] <= 0) return TF_E_RANGE;
    for (int i = 0; i < n; ++i) p->refcnt[ids[i]]++;
    return TF_OK;
}

extern "C" int tf_kvpool_release(tf_kvpool *p, const int32_t *ids, int32_t n) {
    if (!p || n < 0 || (n > 0 && !ids)) return TF_E_ARG;
    std::lock_guard<std::mutex> g(p->mu);
    // check first (a repeated id must hold as many references as it appears)
    std::vector<int32_t> need;
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= p->desc.num_pages) return TF_E_RANGE;
        need.push_back(ids[i]);
    }
    std::vector<int32_t> cnt(p->refcnt);
    for (int32_t id : need)
        if (--cnt[id] < 0) return TF_E_RANGE;
    const size_t N = p->free_ring.size();
    for (int32_t id : need) {
        if (--p->refcnt[id] == 0) {
            p->free_ring[(p->free_head + p->free_count) % N] = id;
            p->free_count++;
        }
    }
    return TF_OK;
}

extern "C" int32_t tf_kvpool_free_pages(const tf_kvpool *p) { return p ? (int32_t)p->free_count : -1; }

extern "C" int32_t tf_kvpool_refcount(const tf_kvpool *p, int32_t id) {
    if (!p || id < 0 || id >= p->desc.num_pages) return -1;
    return p->refcnt[id];
}

extern "C" void *tf_kvpool_page_ptr(const tf_kvpool *p, int32_t cache, int32_t page) {
    if (!p || cache < 0 || cache >= p->desc.num_caches || page < 0 || page >= p->desc.num_pages) return nullptr;
    return p->base + ((size_t)cache * p->desc.num_pages + page) * page_bytes(p->desc);
}

// ---- plan (issue #1313, "Why" bullet 3 and "Proposal" step 1.1) ----
extern "C" int tf_kvpool_plan(const tf_plan_in *in, tf_plan_out *out) {
    if (!in || !out) return TF_E_ARG;
    if (in->room_bytes < 0 || in->context_tokens < 1 || in->lanes < 1 || in->page_rows < 1 || in->lookahead < 0 ||
        in->bytes_per_token < 1 || in->fixed_bytes < 0 || in->cache_budget_bytes < 0)
        return TF_E_ARG;
    const __int128 page_bytes = (__int128)in->page_rows * in->bytes_per_token;
    const int64_t wpages = (in->context_tokens + in->lookahead + in->page_rows - 1) / in->page_rows;
    const __int128 wbytes = (__int128)wpages * page_bytes;
    int64_t n = 1;
    if (in->engine_paged) {
        __int128 spare = (__int128)in->room_bytes - wbytes;
        if (spare > 0) n = 1 + (int64_t)(spare / (wbytes + in->fixed_bytes));
        if (n > in->lanes) n = in->lanes;
        if (n < 1) n = 1;
    }
    int64_t stream_pages = n * wpages;
    if (wpages + (in->lanes - 1) > stream_pages) stream_pages = wpages + (in->lanes - 1);
    const __int128 charged = (__int128)stream_pages * page_bytes + (__int128)(in->lanes - 1) * in->fixed_bytes;
    if (charged > in->room_bytes) return TF_E_NOMEM;
    __int128 left = (__int128)in->room_bytes - charged;
    __int128 cache = left < in->cache_budget_bytes ? left : (__int128)in->cache_budget_bytes;
    int64_t other = (int64_t)((left - cache) / page_bytes);
    out->n_windows = (int32_t)n;
    out->window_pages = wpages;
    out->stream_pages = stream_pages;
    out->cache_bytes = (int64_t)cache;
    out->other_pages = other;
    out->pool_pages = stream_pages + other;
    out->pool_tokens = out->pool_pages * in->page_rows;
    return TF_OK;
}

// ---- paged append ----
extern "C" int tf_paged_append(tf_kvpool *p, int32_t cache, const int32_t *d_pt, int32_t max_pages,
                               const int64_t *h_pos, int32_t S, int32_t n, const void *d_latent, const void *d_rope,
                               void *stream) {
    if (!p || !h_pos || S < 1 || S > TF_MAX_STREAMS || n < 0 || max_pages < 1) return TF_E_ARG;
    if (n > 0 && (!d_latent || !d_rope)) return TF_E_ARG;
    if (cache < 0 || cache >= p->desc.num_caches) return TF_E_RANGE;
    if (!d_pt && (int64_t)S * max_pages > p->desc.num_pages) return TF_E_RANGE;
    for (int s = 0; s < S; ++s)
        if (h_pos[s] < 0 || h_pos[s] > (int64_t)max_pages * kPageRows - n) return TF_E_RANGE;
    if (n == 0) return TF_OK;
    if (is_fp8(p->desc))
        return launch_append_fp8(p, cache, d_pt, max_pages, h_pos, S, n, d_latent, d_rope, (cudaStream_t)stream);
    return launch_append(p, cache, d_pt, max_pages, h_pos, S, n, d_latent, d_rope, (cudaStream_t)stream);
}

// ---- attention ----
// The launch numbers a stream's rows and key tiles in int32 (and listed rows are int32), so a
// stream may hold at most INT32_MAX rows.  Only a table that repeats page ids can describe more.
static constexpr int64_t kMaxStreamRows = INT32_MAX;

extern "C" size_t tf_paged_mla_workspace_bytes(const tf_kvpool *p, int32_t S, int32_t R, int32_t H,
                                               const int64_t *h_len) {
    if (S < 1 || S > TF_MAX_STREAMS || R < 1 || H < 1 || H > TF_MAX_HEADS || !h_len) return 0;
    if ((int64_t)S * R * H > (int64_t)1 << 30) return 0;   // refused by tf_paged_mla_attend
    for (int s = 0; s < S; ++s)
        if (h_len[s] < R || h_len[s] > kMaxStreamRows) return 0;
    const bool invariant = p && (p->desc.flags & TF_POOL_BATCH_INVARIANT);
    const size_t part = attend_workspace_bytes(invariant, S, R, H, h_len);
    // FP8 pages on a batch-invariant pool are expanded to bf16 in the workspace first
    if (p && is_fp8(p->desc) && invariant) return (part + 1023) / 1024 * 1024 + fp8_shadow_bytes(S, h_len);
    return part;
}

extern "C" int tf_paged_mla_plan_info(int32_t S, int32_t R, int32_t H, const int64_t *h_len, int32_t sms,
                                      int32_t invariant, tf_attend_plan *info, int64_t *range_bounds,
                                      int64_t *split_keys) {
    if (!h_len || !info || S < 1 || S > TF_MAX_STREAMS || R < 1 || H < 1 || H > TF_MAX_HEADS) return TF_E_ARG;
    if ((int64_t)S * R * H > (int64_t)1 << 30) return TF_E_UNSUPPORTED;   // as tf_paged_mla_attend
    for (int s = 0; s < S; ++s)
        if (h_len[s] < R || h_len[s] > kMaxStreamRows) return TF_E_RANGE;
    return attend_plan_info(S, R, H, h_len, sms, invariant != 0, info, range_bounds, split_keys);
}

extern "C" int tf_paged_mla_attend(tf_kvpool *p, int32_t cache, const int32_t *d_pt, int32_t max_pages,
                                   const int64_t *h_len, int32_t S, int32_t R, int32_t H, const void *d_q,
                                   float scale, void *d_out, float *d_lse, void *d_ws, size_t ws_bytes,
                                   void *stream) {
    if (!p || !h_len || !d_q || !d_out || S < 1 || S > TF_MAX_STREAMS || R < 1 || H < 1 || H > TF_MAX_HEADS ||
        max_pages < 1)
        return TF_E_ARG;
    if (!(scale > 0.0f) || scale == 1.0f / 0.0f) return TF_E_ARG;
    if (cache < 0 || cache >= p->desc.num_caches) return TF_E_RANGE;
    if (!d_pt && (int64_t)S * max_pages > p->desc.num_pages) return TF_E_RANGE;
    if ((int64_t)S * R * H > (int64_t)1 << 30) return TF_E_UNSUPPORTED;
    for (int s = 0; s < S; ++s)
        if (h_len[s] < R || h_len[s] > (int64_t)max_pages * kPageRows) return TF_E_RANGE;
    for (int s = 0; s < S; ++s)
        if (h_len[s] > kMaxStreamRows) return TF_E_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(d_q) & 15u) != 0 || (reinterpret_cast<uintptr_t>(d_out) & 15u) != 0)
        return TF_E_ARG;
    const bool invariant = (p->desc.flags & TF_POOL_BATCH_INVARIANT) != 0;
    const size_t part = attend_workspace_bytes(invariant, S, R, H, h_len);
    const bool expand = is_fp8(p->desc) && invariant;   // else FP8 codes are expanded in the kernel
    const size_t need = expand ? (part + 1023) / 1024 * 1024 + fp8_shadow_bytes(S, h_len) : part;
    if (need > 0 && (!d_ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(d_ws) & 255u) != 0))
        return d_ws && ws_bytes < need ? TF_E_NOMEM : TF_E_ARG;
    if (expand)
        return launch_attend_fp8(p, cache, d_pt, max_pages, h_len, S, R, H, d_q, scale, d_out, d_lse, d_ws, ws_bytes,
                                 part, (cudaStream_t)stream);
    return launch_attend(p, cache, d_pt, max_pages, h_len, S, R, H, d_q, scale, d_out, d_lse, d_ws, ws_bytes,
                         (cudaStream_t)stream);
}

// ---- kept-state copy ----
// ---- attention over listed rows ----
static int sparse_checks(const tf_kvpool *p, int32_t S, int32_t H, int32_t max_idx, const int32_t *h_nidx) {
    if (S < 1 || S > TF_MAX_STREAMS || H < 1 || H > TF_MAX_HEADS || max_idx < 1 || !h_nidx) return TF_E_ARG;
    for (int s = 0; s < S; ++s)
        if (h_nidx[s] < 1 || h_nidx[s] > max_idx) return TF_E_RANGE;
    // the gather views number pool rows in int32 (4,608 rope rows a page)
    if (p && (int64_t)p->desc.num_caches * p->desc.num_pages * (int64_t)(kPageBytes / (kRope * 2)) >= ((int64_t)1 << 31))
        return TF_E_UNSUPPORTED;
    return TF_OK;
}

extern "C" size_t tf_paged_mla_sparse_workspace_bytes(const tf_kvpool *p, int32_t S, int32_t H, const int32_t *h_nidx) {
    if (sparse_checks(p, S, H, h_nidx ? 1 << 30 : 1, h_nidx) != TF_OK) return 0;
    int64_t n[TF_MAX_STREAMS];
    for (int s = 0; s < S; ++s) n[s] = h_nidx[s];
    return attend_workspace_bytes(false, S, 1, H, n, true);
}

extern "C" int tf_paged_mla_attend_sparse(tf_kvpool *p, int32_t cache, const int32_t *d_pt, int32_t max_pages,
                                          const int64_t *h_len, const int32_t *d_idx, int32_t max_idx,
                                          const int32_t *h_nidx, int32_t S, int32_t H, const void *d_q, float scale,
                                          void *d_out, float *d_lse, void *d_ws, size_t ws_bytes, void *stream) {
    if (!p || !h_len || !d_idx || !d_q || !d_out || max_pages < 1) return TF_E_ARG;
    const int rc = sparse_checks(p, S, H, max_idx, h_nidx);
    if (rc != TF_OK) return rc;
    if (!(scale > 0.0f) || scale == 1.0f / 0.0f) return TF_E_ARG;
    if (cache < 0 || cache >= p->desc.num_caches) return TF_E_RANGE;
    if (!d_pt && (int64_t)S * max_pages > p->desc.num_pages) return TF_E_RANGE;
    for (int s = 0; s < S; ++s)
        if (h_len[s] < 1 || h_len[s] > (int64_t)max_pages * kPageRows) return TF_E_RANGE;
    for (int s = 0; s < S; ++s)
        if (h_len[s] > kMaxStreamRows) return TF_E_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(d_q) & 15u) != 0 || (reinterpret_cast<uintptr_t>(d_out) & 15u) != 0)
        return TF_E_ARG;
    int64_t n[TF_MAX_STREAMS];
    for (int s = 0; s < S; ++s) n[s] = h_nidx[s];
    const size_t need = attend_workspace_bytes(false, S, 1, H, n, true);
    if (need > 0 && (!d_ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(d_ws) & 255u) != 0))
        return d_ws && ws_bytes < need ? TF_E_NOMEM : TF_E_ARG;
    return launch_attend(p, cache, d_pt, max_pages, h_len, S, 1, H, d_q, scale, d_out, d_lse, d_ws, ws_bytes,
                         (cudaStream_t)stream, d_idx, max_idx, h_nidx);
}

extern "C" int tf_state_copy_rows(tf_kvpool *p, int32_t cache, const int32_t *d_src, const int32_t *d_dst,
                                  int64_t at, void *stream) {
    if (!p || at < 0) return TF_E_ARG;
    if (cache >= p->desc.num_caches) return TF_E_RANGE;
    if (at > (int64_t)p->desc.num_pages * kPageRows) return TF_E_RANGE;
    if (at == 0) return TF_OK;
    if (!d_src || !d_dst) return TF_E_ARG;
    if (is_fp8(p->desc)) return launch_state_copy_fp8(p, cache, d_src, d_dst, at, (cudaStream_t)stream);
    return launch_state_copy(p, cache, d_src, d_dst, at, (cudaStream_t)stream);
}

// ---- diagnostics ----
extern "C" int tf_last_error(tf_kvpool *p, int64_t *detail) {
    if (!p) return TF_E_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return TF_E_CUDA;
    DevErr e{};
    if (cudaMemcpy(&e, p->err, sizeof e, cudaMemcpyDeviceToHost) != cudaSuccess) return TF_E_CUDA;
    if (cudaMemset(p->err, 0, sizeof(DevErr)) != cudaSuccess) return TF_E_CUDA;
    if (!p->err_cleared.load()) e = DevErr{};  // nothing launched yet: the word was never zeroed
    p->err_cleared.store(true);
    if (detail) *detail = e.detail;
    return e.code;
}

extern "C" int tf_diag_wait_timeout(tf_kvpool *p, int64_t limit_cycles, void *stream) {
    if (!p || limit_cycles < 1 || limit_cycles > (int64_t(1) << 32)) return TF_E_ARG;
    return launch_diag_wait(p, (long long)limit_cycles, (cudaStream_t)stream);
}

extern "C" int64_t tf_launch_count(void) { return launch_counter().load(); }

extern "C" int tf_profile_enable(tf_kvpool *p, int32_t on) {
    if (!p) return TF_E_ARG;
    p->prof = on != 0;
    return TF_OK;
}

extern "C" int tf_profile_read(tf_kvpool *p, int32_t kind, double *total_ms, int64_t *launches) {
    if (!p || kind < 0 || kind >= kProfKinds) return TF_E_ARG;
    std::lock_guard<std::mutex> g(p->mu);
    double tot = 0.0;
    int64_t cnt = 0;
    std::vector<ProfRec> keep;
    for (auto &r : p->recs) {
        if (r.kind != kind) {
            keep.push_back(r);
            continue;
        }
        if (cudaEventSynchronize(r.b) != cudaSuccess) return TF_E_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return TF_E_CUDA;
        tot += ms;
        cnt++;
        p->spare_events.push_back(r.a);
        p->spare_events.push_back(r.b);
    }
    p->recs.swap(keep);
    if (total_ms) *total_ms = tot;
    if (launches) *launches = cnt;
    return TF_OK;
}
