// Row-moving kernels: the paged append (issue #1142, piece 2: the row-writing
// kernel takes the page table), the kept-state copy (issue #1142, piece 1: copy
// each cache's first `at` rows) and the poison fill of taken pages (TF_KV_POISON,
// same page).  All three move bytes only, 16 at a time, and are bounded by HBM.
#include "ptx.cuh"
#include "tf_internal.h"

namespace tf {

struct AppendParams {
    const int32_t *pt;   // [S][max_pages] or null (windows)
    const uint4 *lat;    // [S][n][512] bf16 = 64 uint4 a row
    const uint4 *rope;   // [S][n][64] bf16 = 8 uint4 a row
    char *cache_base;    // page 0 of this cache
    DevErr *err;
    int32_t max_pages, num_pages, S, n;
    int64_t pos[TF_MAX_STREAMS];
};

// One warp per new row: 64 + 8 16-byte chunks.
__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendParams p) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= (int64_t)p.S * p.n) return;
    const int s = (int)(row / p.n);
    const int i = (int)(row - (int64_t)s * p.n);
    const int64_t pos = p.pos[s] + i;
    const int lp = (int)(pos >> 9), r = (int)(pos & 511);
    const int page = p.pt ? __ldg(p.pt + (int64_t)s * p.max_pages + lp) : s * p.max_pages + lp;
    if (page < 0 || page >= p.num_pages) {
        if (lane == 0) ptx::record_error(p.err, TF_E_DEVICE, page);
        return;
    }
    char *pg = p.cache_base + (size_t)page * kPageBytes;
    uint4 *dl = reinterpret_cast<uint4 *>(pg + (size_t)r * (kLat * 2));
    const uint4 *sl = p.lat + row * 64;
    uint4 a = __ldg(sl + lane), b = __ldg(sl + lane + 32);
    dl[lane] = a;
    dl[lane + 32] = b;
    if (lane < 8) {
        uint4 *dr = reinterpret_cast<uint4 *>(pg + kLatBlockBytes + (size_t)r * (kRope * 2));
        dr[lane] = __ldg(p.rope + row * 8 + lane);
    }
}

int launch_append(tf_kvpool *pool, int cache, const int32_t *d_pt, int max_pages, const int64_t *h_pos, int S, int n,
                  const void *d_lat, const void *d_rope, cudaStream_t st) {
    AppendParams p;
    p.pt = d_pt;
    p.lat = static_cast<const uint4 *>(d_lat);
    p.rope = static_cast<const uint4 *>(d_rope);
    p.cache_base = pool->base + (size_t)cache * pool->desc.num_pages * kPageBytes;
    p.err = pool->err;
    p.max_pages = max_pages;
    p.num_pages = pool->desc.num_pages;
    p.S = S;
    p.n = n;
    for (int s = 0; s < S; ++s) p.pos[s] = h_pos[s];
    if ((reinterpret_cast<uintptr_t>(d_lat) & 15u) || (reinterpret_cast<uintptr_t>(d_rope) & 15u)) return TF_E_ARG;
    const int64_t rows = (int64_t)S * n;
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 0x7FFFFFFF) return TF_E_UNSUPPORTED;
    if (prepare_launch(pool, st) != TF_OK) return TF_E_CUDA;
    ProfScope prof(pool, kProfAppend, st);
    const cudaError_t e = launch_pdl(append_kernel, dim3((unsigned)blocks), dim3(256), 0, st, p);
    launch_counter()++;
    return e == cudaSuccess ? TF_OK : TF_E_CUDA;
}

// One block per (page of the state, cache): the latent rows [0, rows) are one
// contiguous run of rows*1 KiB, the rope rows one run of rows*128 B.
__global__ void __launch_bounds__(512) state_copy_kernel(char *base, int num_pages, int cache0,
                                                         const int32_t *__restrict__ src,
                                                         const int32_t *__restrict__ dst, int64_t at, DevErr *err) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    const int pg = blockIdx.x;
    const int cache = cache0 + blockIdx.y;
    const int64_t rem = at - (int64_t)pg * kPageRows;
    const int rows = rem < kPageRows ? (int)rem : kPageRows;
    const int sp = __ldg(src + pg), dp = __ldg(dst + pg);
    if (sp < 0 || sp >= num_pages || dp < 0 || dp >= num_pages) {
        if (threadIdx.x == 0) ptx::record_error(err, TF_E_DEVICE, (sp < 0 || sp >= num_pages) ? sp : dp);
        return;
    }
    char *cbase = base + (size_t)cache * num_pages * kPageBytes;
    const uint4 *s = reinterpret_cast<const uint4 *>(cbase + (size_t)sp * kPageBytes);
    uint4 *d = reinterpret_cast<uint4 *>(cbase + (size_t)dp * kPageBytes);
    const int nl = rows * (kLat * 2 / 16), nr = rows * (kRope * 2 / 16);
    const int rope_off = (int)(kLatBlockBytes / 16);
    const int total = nl + nr;
    constexpr int U = 4;
    for (int k0 = threadIdx.x; k0 < total; k0 += blockDim.x * U) {
        uint4 v[U];
        int off[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            int k = k0 + u * blockDim.x;
            off[u] = k < nl ? k : rope_off + (k - nl);
            if (k < total) v[u] = __ldg(s + off[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (k0 + u * (int)blockDim.x < total) d[off[u]] = v[u];
    }
}

int launch_state_copy(tf_kvpool *pool, int cache, const int32_t *d_src, const int32_t *d_dst, int64_t at,
                      cudaStream_t st) {
    const int64_t pages = (at + kPageRows - 1) / kPageRows;
    const int c0 = cache < 0 ? 0 : cache;
    const int nc = cache < 0 ? pool->desc.num_caches : 1;
    dim3 grid((unsigned)pages, (unsigned)nc);
    if (prepare_launch(pool, st) != TF_OK) return TF_E_CUDA;
    ProfScope prof(pool, kProfCopy, st);
    const cudaError_t e = launch_pdl(state_copy_kernel, grid, dim3(512), 0, st, pool->base, pool->desc.num_pages, c0,
                                     d_src, d_dst, at, pool->err);
    launch_counter()++;
    return e == cudaSuccess ? TF_OK : TF_E_CUDA;
}

constexpr int kPoisonIds = 2048;
struct PoisonParams {
    char *base;
    size_t page_bytes;   // a multiple of 256
    uint32_t pattern;    // the fill word: bf16 NaN pairs, or all ones on FP8 pages
    int32_t num_pages, num_caches, n;
    int32_t ids[kPoisonIds];
};

// grid (ids, caches, 16 slices of a page): fill with the pattern (bf16 NaN 0x7FC0 pairs on BF16
// pages; 0xFF bytes on FP8 pages, NaN as codes, scales and rope alike).
__global__ void __launch_bounds__(256) poison_kernel(const __grid_constant__ PoisonParams p) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    const int id = p.ids[blockIdx.x];
    const int cache = blockIdx.y;
    uint4 *pg = reinterpret_cast<uint4 *>(p.base + ((size_t)cache * p.num_pages + id) * p.page_bytes);
    const int per_slice = (int)(p.page_bytes / 16 / 16);
    const uint4 nan4 = make_uint4(p.pattern, p.pattern, p.pattern, p.pattern);
    uint4 *q = pg + (size_t)blockIdx.z * per_slice;
    for (int k = threadIdx.x; k < per_slice; k += blockDim.x) q[k] = nan4;
}

int launch_poison(tf_kvpool *pool, const int32_t *h_ids, int n, cudaStream_t st) {
    if (prepare_launch(pool, st) != TF_OK) return TF_E_CUDA;
    for (int b = 0; b < n; b += kPoisonIds) {
        PoisonParams p;
        p.base = pool->base;
        p.page_bytes = page_bytes(pool->desc);
        p.pattern = is_fp8(pool->desc) ? 0xFFFFFFFFu : 0x7FC07FC0u;
        p.num_pages = pool->desc.num_pages;
        p.num_caches = pool->desc.num_caches;
        p.n = std::min(kPoisonIds, n - b);
        for (int i = 0; i < p.n; ++i) p.ids[i] = h_ids[b + i];
        dim3 grid((unsigned)p.n, (unsigned)p.num_caches, 16);
        ProfScope prof(pool, kProfPoison, st);
        const cudaError_t e = launch_pdl(poison_kernel, grid, dim3(256), 0, st, p);
        launch_counter()++;
        if (e != cudaSuccess) return TF_E_CUDA;
    }
    return TF_OK;
}

// One block waits on a barrier that nothing completes; the bounded wait must give up.
__global__ void diag_wait_kernel(DevErr *err, long long limit) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) ptx::mbar_wait(&bar, 0, &abort_flag, err, 99, limit);
}

int launch_diag_wait(tf_kvpool *pool, long long limit, cudaStream_t st) {
    if (prepare_launch(pool, st) != TF_OK) return TF_E_CUDA;
    diag_wait_kernel<<<1, 32, 0, st>>>(pool->err, limit);
    launch_counter()++;
    return cudaGetLastError() == cudaSuccess ? TF_OK : TF_E_CUDA;
}

}  // namespace tf
