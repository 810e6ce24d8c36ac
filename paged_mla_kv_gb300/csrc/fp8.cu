// FP8 pages (issue #1313, step 1.3, item 3: FP8 latent rows on pages, a page's fp32 row scales
// stored behind its rows; windows laid out the same way, under the same addressing rule).  A page of one cache: 512 x 512 E4M3 codes, 512 fp32 scales, 512 x 64 bf16 rope.
//
// append_fp8_kernel quantizes each new latent row (amax / 448 scale, E4M3 round-to-nearest-even
// with saturation); state_copy_fp8_kernel copies the first `at` rows of a kept state block by
// block.  The attention kernel reads the codes itself (attend.cu); on a batch-invariant pool
// the rows are first expanded to bf16 pages in the caller's workspace (dequant_kernel) and the
// BF16 attention runs over that view.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <mutex>

#include "ptx.cuh"
#include "tf_internal.h"

namespace tf {

struct AppendFp8Params {
    const int32_t *pt;   // [S][max_pages] or null (windows)
    const uint4 *lat;    // [S][n][512] bf16 = 64 uint4 a row
    const uint4 *rope;   // [S][n][64] bf16 = 8 uint4 a row
    char *cache_base;    // page 0 of this cache
    DevErr *err;
    int32_t max_pages, num_pages, S, n;
    int64_t pos[TF_MAX_STREAMS];
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One warp per new row; lane l quantizes latent values 16l .. 16l + 15.
__global__ void __launch_bounds__(256) append_fp8_kernel(const __grid_constant__ AppendFp8Params p) {
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
    const uint4 a = __ldg(p.lat + row * 64 + 2 * lane), b = __ldg(p.lat + row * 64 + 2 * lane + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float x[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        x[2 * k] = bf16_lo(w[k]);
        x[2 * k + 1] = bf16_hi(w[k]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(amax, 448.0f);
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
    if (amax > 0.0f) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint32_t c = __nv_cvt_float_to_fp8(__fdiv_rn(x[k], scale), __NV_SATFINITE, __NV_E4M3);
            packed[k >> 2] |= c << (8 * (k & 3));
        }
    }
    char *pg = p.cache_base + (size_t)page * kF8PageBytes;
    reinterpret_cast<uint4 *>(pg + (size_t)r * kLat)[lane] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if (lane == 0) reinterpret_cast<float *>(pg + kF8ScaleOff)[r] = scale;
    if (lane < 8) reinterpret_cast<uint4 *>(pg + kF8RopeOff + (size_t)r * (kRope * 2))[lane] = __ldg(p.rope + row * 8 + lane);
}

// One block per (page of the state, cache): codes rows x 512 B, scales rows x 4 B, rope
// rows x 128 B; nothing at or past row `at`.
__global__ void __launch_bounds__(512) state_copy_fp8_kernel(char *base, int num_pages, int cache0,
                                                             const int32_t *__restrict__ src,
                                                             const int32_t *__restrict__ dst, int64_t at,
                                                             DevErr *err) {
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
    char *cbase = base + (size_t)cache * num_pages * kF8PageBytes;
    const char *s = cbase + (size_t)sp * kF8PageBytes;
    char *d = cbase + (size_t)dp * kF8PageBytes;
    const int nc = rows * (kLat / 16), nr = rows * (kRope * 2 / 16);
    for (int k = threadIdx.x; k < nc; k += blockDim.x)
        reinterpret_cast<uint4 *>(d)[k] = __ldg(reinterpret_cast<const uint4 *>(s) + k);
    for (int k = threadIdx.x; k < rows; k += blockDim.x)
        reinterpret_cast<uint32_t *>(d + kF8ScaleOff)[k] = __ldg(reinterpret_cast<const uint32_t *>(s + kF8ScaleOff) + k);
    for (int k = threadIdx.x; k < nr; k += blockDim.x)
        reinterpret_cast<uint4 *>(d + kF8RopeOff)[k] = __ldg(reinterpret_cast<const uint4 *>(s + kF8RopeOff) + k);
}

struct DequantParams {
    const char *cache_base;  // FP8 page 0 of this cache
    const int32_t *pt;       // [S][max_pages] or null (windows)
    char *shadow;            // BF16 pages
    int32_t *shadow_pt;      // [S][maxp]
    DevErr *err;
    int32_t max_pages, num_pages, S, maxp;
    int64_t len[TF_MAX_STREAMS];
    int32_t off[TF_MAX_STREAMS];  // the stream's first shadow page
};

// grid (maxp, S): logical page j of stream s, rows [0, min(512, len - 512 j)), expanded to a
// BF16 page: latent value = bf16(code * scale), rope copied.
constexpr int kDequantThreads = 512;

__global__ void __launch_bounds__(kDequantThreads) dequant_kernel(const __grid_constant__ DequantParams p) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    const int j = blockIdx.x, s = blockIdx.y;
    const int64_t rem = p.len[s] - (int64_t)j * kPageRows;
    if (rem <= 0) return;
    const int rows = rem < kPageRows ? (int)rem : kPageRows;
    const int page = p.pt ? __ldg(p.pt + (int64_t)s * p.max_pages + j) : s * p.max_pages + j;
    if (page < 0 || page >= p.num_pages) {
        if (threadIdx.x == 0) ptx::record_error(p.err, TF_E_DEVICE, page);
        return;
    }
    const int dpage = p.off[s] + j;
    if (threadIdx.x == 0) p.shadow_pt[(int64_t)s * p.maxp + j] = dpage;
    const char *src = p.cache_base + (size_t)page * kF8PageBytes;
    char *dst = p.shadow + (size_t)dpage * kPageBytes;
    const float *scales = reinterpret_cast<const float *>(src + kF8ScaleOff);
    const int nc = rows * (kLat / 16);  // 16 codes a unit
    constexpr int U = 4;                // units a thread has in flight
    for (int k0 = threadIdx.x; k0 < nc; k0 += U * kDequantThreads) {
        uint4 c[U];
        float sc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int k = k0 + u * kDequantThreads;
            if (k < nc) {
                c[u] = __ldg(reinterpret_cast<const uint4 *>(src) + k);
                sc[u] = __ldg(scales + (k >> 5));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int k = k0 + u * kDequantThreads;
            if (k >= nc) break;
            const uint32_t cw[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
            uint32_t o[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
                        (__nv_fp8x2_storage_t)((cw[q] >> (16 * h)) & 0xFFFFu), __NV_E4M3);
                    const float2 f = __half22float2(__half2(hr));
                    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * sc[u], f.y * sc[u]);
                    o[2 * q + h] = *reinterpret_cast<const uint32_t *>(&b);
                }
            }
            uint4 *d = reinterpret_cast<uint4 *>(dst) + 2 * k;
            d[0] = make_uint4(o[0], o[1], o[2], o[3]);
            d[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
    }
    const int nr = rows * (kRope * 2 / 16);
    for (int k = threadIdx.x; k < nr; k += blockDim.x)
        reinterpret_cast<uint4 *>(dst + kLatBlockBytes)[k] = __ldg(reinterpret_cast<const uint4 *>(src + kF8RopeOff) + k);
}

int launch_append_fp8(tf_kvpool *pool, int cache, const int32_t *d_pt, int max_pages, const int64_t *h_pos, int S,
                      int n, const void *d_lat, const void *d_rope, cudaStream_t st) {
    if ((reinterpret_cast<uintptr_t>(d_lat) & 15u) || (reinterpret_cast<uintptr_t>(d_rope) & 15u)) return TF_E_ARG;
    AppendFp8Params p;
    p.pt = d_pt;
    p.lat = static_cast<const uint4 *>(d_lat);
    p.rope = static_cast<const uint4 *>(d_rope);
    p.cache_base = pool->base + (size_t)cache * pool->desc.num_pages * kF8PageBytes;
    p.err = pool->err;
    p.max_pages = max_pages;
    p.num_pages = pool->desc.num_pages;
    p.S = S;
    p.n = n;
    for (int s = 0; s < S; ++s) p.pos[s] = h_pos[s];
    const int64_t blocks = ((int64_t)S * n + 7) / 8;
    if (blocks > 0x7FFFFFFF) return TF_E_UNSUPPORTED;
    if (prepare_launch(pool, st) != TF_OK) return TF_E_CUDA;
    ProfScope prof(pool, kProfAppend, st);
    const cudaError_t e = launch_pdl(append_fp8_kernel, dim3((unsigned)blocks), dim3(256), 0, st, p);
    launch_counter()++;
    return e == cudaSuccess ? TF_OK : TF_E_CUDA;
}

int launch_state_copy_fp8(tf_kvpool *pool, int cache, const int32_t *d_src, const int32_t *d_dst, int64_t at,
                          cudaStream_t st) {
    const int64_t pages = (at + kPageRows - 1) / kPageRows;
    const int c0 = cache < 0 ? 0 : cache;
    const int nc = cache < 0 ? pool->desc.num_caches : 1;
    if (prepare_launch(pool, st) != TF_OK) return TF_E_CUDA;
    ProfScope prof(pool, kProfCopy, st);
    const cudaError_t e = launch_pdl(state_copy_fp8_kernel, dim3((unsigned)pages, (unsigned)nc), dim3(512), 0, st,
                                     pool->base, pool->desc.num_pages, c0, d_src, d_dst, at, pool->err);
    launch_counter()++;
    return e == cudaSuccess ? TF_OK : TF_E_CUDA;
}

namespace {
struct ShadowPlan {
    int64_t pages = 0;   // BF16 pages over all streams
    int32_t maxp = 0;    // most pages of one stream
    size_t table_bytes = 0;
};
ShadowPlan shadow_plan(int S, const int64_t *h_len) {
    ShadowPlan sp;
    for (int s = 0; s < S; ++s) {
        const int64_t np = (h_len[s] + kPageRows - 1) / kPageRows;
        sp.pages += np;
        sp.maxp = std::max<int32_t>(sp.maxp, (int32_t)np);
    }
    sp.table_bytes = ((size_t)S * sp.maxp * 4 + 1023) / 1024 * 1024;
    return sp;
}
}  // namespace

// The expanded rows: a page table and the BF16 pages, with room to align the pages to 1 KiB.
size_t fp8_shadow_bytes(int S, const int64_t *h_len) {
    const ShadowPlan sp = shadow_plan(S, h_len);
    return sp.table_bytes + 1024 + (size_t)sp.pages * kPageBytes;
}

int launch_attend_fp8(tf_kvpool *pool, int cache, const int32_t *d_pt, int max_pages, const int64_t *h_len, int S,
                      int R, int H, const void *d_q, float scale, void *d_out, float *d_lse, void *d_ws,
                      size_t ws_bytes, size_t attend_ws, cudaStream_t st) {
    const ShadowPlan sp = shadow_plan(S, h_len);
    if (sp.pages * (int64_t)kPageBytes / (int64_t)kPageBytes != sp.pages || sp.pages >= (1ll << 31))
        return TF_E_UNSUPPORTED;
    const size_t part = (attend_ws + 1023) / 1024 * 1024;  // partials first, as on a BF16 pool
    char *ws = static_cast<char *>(d_ws);
    int32_t *spt = reinterpret_cast<int32_t *>(ws + part);
    const uintptr_t raw = reinterpret_cast<uintptr_t>(ws + part + sp.table_bytes);
    char *shadow = reinterpret_cast<char *>((raw + 1023) & ~uintptr_t(1023));
    if ((size_t)(shadow - ws) + (size_t)sp.pages * kPageBytes > ws_bytes) return TF_E_NOMEM;

    // the BF16 view over the workspace: one cache, its own maps, the pool's error word; held
    // until both launches are queued (their parameters are copied at launch)
    std::lock_guard<std::mutex> guard(pool->shadow_mu);
    tf_kvpool *sh = pool->shadow;
    if (!sh) {
        sh = new (std::nothrow) tf_kvpool();
        if (!sh) return TF_E_NOMEM;
        pool->shadow = sh;
    }
    if (sh->base != shadow || sh->desc.num_pages != (int32_t)sp.pages) sh->tmaps_ready = false;
    sh->desc = pool->desc;
    sh->desc.num_caches = 1;
    sh->desc.num_pages = (int32_t)sp.pages;
    sh->desc.flags = pool->desc.flags & TF_POOL_BATCH_INVARIANT;
    sh->base = shadow;
    sh->bytes = (size_t)sp.pages * kPageBytes;
    sh->err = pool->err;
    sh->err_cleared.store(true);
    sh->prof = false;

    DequantParams p;
    p.cache_base = pool->base + (size_t)cache * pool->desc.num_pages * kF8PageBytes;
    p.pt = d_pt;
    p.shadow = shadow;
    p.shadow_pt = spt;
    p.err = pool->err;
    p.max_pages = max_pages;
    p.num_pages = pool->desc.num_pages;
    p.S = S;
    p.maxp = sp.maxp;
    int32_t off = 0;
    for (int s = 0; s < S; ++s) {
        p.len[s] = h_len[s];
        p.off[s] = off;
        off += (int32_t)((h_len[s] + kPageRows - 1) / kPageRows);
    }
    if (prepare_launch(pool, st) != TF_OK) return TF_E_CUDA;
    ProfScope prof(pool, kProfAttend, st);  // the expansion and the attention together
    const cudaError_t e =
        launch_pdl(dequant_kernel, dim3((unsigned)sp.maxp, (unsigned)S), dim3(kDequantThreads), 0, st, p);
    launch_counter()++;
    if (e != cudaSuccess) return TF_E_CUDA;
    return launch_attend(sh, 0, spt, sp.maxp, h_len, S, R, H, d_q, scale, d_out, d_lse, d_ws, attend_ws, st);
}

}  // namespace tf
