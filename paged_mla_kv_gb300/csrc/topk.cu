// Blocked top-k with an exact merge ("Running CHUNKED_PREFILL_SIZE above 1024 without the
// long-prompt memory problem", section 2.3): every block of a row keeps its top-k, the top-k of
// the candidates is the row's top-k.  Order: the IEEE total order of fp32 (a NaN below every
// number), larger first, ties by the smaller column.
//
// One CTA a block.  The block's keys live in registers (32 a thread for logits, 16 key/column
// pairs a thread for candidates), mapped to unsigned integers that compare like the values.
// A radix select with digits of 11, 11 and 10 bits (histograms in shared memory) finds the
// k-th key; it stops early at the first digit whose bin is needed whole.  When only part of the
// keys equal to the k-th are needed, a second radix select over their columns picks the
// smallest.  The winners are compacted with one shared atomic a warp; the last level sorts
// them (bitonic, in shared memory) and writes columns and values.
#include <cstdint>

#include "../../include/tf_topk.h"
#include "ptx.cuh"
#include "tf_internal.h"

namespace tf {
namespace topk {

constexpr int T = 512;
constexpr int E0 = TF_TOPK_BLOCK / T;  // 32 logits a thread
constexpr int E1 = TF_TOPK_MERGE / T;  // 16 candidates a thread
constexpr uint32_t kPad = 0xFFFFFFFFu; // the column of a filler candidate

static_assert(E0 % 4 == 0, "first-level keys are loaded four at a time");

struct Level {
    const float *logits;
    int64_t ld, n;
    const int32_t *len;
    const uint2 *cin;  // candidates in (key, column): cin_row a row
    int64_t cin_row;
    uint2 *cout;       // candidates out: nch * k a row
    int32_t nch, k;
    int32_t *out_idx;
    float *out_val;
};

// fp32 bits -> an unsigned key with the same order (the IEEE total order); every NaN -> 0.
__device__ __forceinline__ uint32_t ord_key(uint32_t u) {
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint32_t key_bits(uint32_t key) {
    return (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
}

struct Bin {
    uint32_t bin, before, count;
};

// Scan the histogram from the best end: the bin in which the cumulative count reaches `want`
// (1 <= want <= total), the count before it and its own count.  DESC: bin nb-1 is the best.
template <bool DESC>
__device__ __forceinline__ Bin find_bin(const uint32_t *hist, int nb, uint32_t want, uint32_t *red) {
    const int per = nb / T;  // 4 or 2
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    uint32_t c[4], s = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        c[j] = 0;
        if (j < per) {
            const int b = DESC ? nb - 1 - (t * per + j) : t * per + j;
            c[j] = hist[b];
            s += c[j];
        }
    }
    uint32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) red[w] = incl;
    __syncthreads();
    if (w == 0) {
        const uint32_t v = lane < T / 32 ? red[lane] : 0u;
        uint32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane < T / 32) red[lane] = x - v;
    }
    __syncthreads();
    uint32_t cum = red[w] + incl - s;
    if (cum < want && want <= cum + s) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < per && cum + c[j] >= want) {
                red[T / 32 + 0] = DESC ? nb - 1 - (t * per + j) : t * per + j;
                red[T / 32 + 1] = cum;
                red[T / 32 + 2] = c[j];
                break;
            }
            cum += c[j];
        }
    }
    __syncthreads();
    return Bin{red[T / 32 + 0], red[T / 32 + 1], red[T / 32 + 2]};
}

// The k-th best key.  Result: every key > lo is taken, and of the keys == lo either all (all)
// or the `rem` with the smallest columns.
template <int E>
__device__ __forceinline__ void key_select(const uint32_t (&key)[E], uint32_t want, uint32_t *hist, uint32_t *red,
                                           uint32_t &lo, uint32_t &rem, bool &all) {
    uint32_t prefix = 0, pmask = 0;
    rem = want;
#pragma unroll 1
    for (int d = 0; d < 3; ++d) {
        const int shift = d == 0 ? 21 : (d == 1 ? 10 : 0);
        const int nb = d == 2 ? 1024 : 2048;
        for (int i = threadIdx.x; i < nb; i += T) hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e)
            if ((key[e] & pmask) == prefix) atomicAdd(&hist[(key[e] >> shift) & (nb - 1)], 1u);
        __syncthreads();
        const Bin r = find_bin<true>(hist, nb, rem, red);
        prefix |= r.bin << shift;
        pmask |= uint32_t(nb - 1) << shift;
        rem -= r.before;
        if (r.count == rem || d == 2) {
            lo = prefix;
            all = r.count == rem;
            return;
        }
    }
}

// Of the keys equal to `lo`, the `want` with the smallest columns: those with column <= the
// returned bound.  Fillers share one column; the caller never lets more than k through.
template <int E, class Col>
__device__ __forceinline__ uint32_t col_select(const uint32_t (&key)[E], Col col, uint32_t lo, uint32_t want,
                                               uint32_t *hist, uint32_t *red) {
    uint32_t prefix = 0, pmask = 0, rem = want;
#pragma unroll 1
    for (int d = 0; d < 3; ++d) {
        const int shift = d == 0 ? 21 : (d == 1 ? 10 : 0);
        const int nb = d == 2 ? 1024 : 2048;
        for (int i = threadIdx.x; i < nb; i += T) hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const uint32_t c = col(e);
            if (key[e] == lo && (c & pmask) == prefix) atomicAdd(&hist[(c >> shift) & (nb - 1)], 1u);
        }
        __syncthreads();
        const Bin r = find_bin<false>(hist, nb, rem, red);
        prefix |= r.bin << shift;
        pmask |= uint32_t(nb - 1) << shift;
        rem -= r.before;
        if (r.count == rem || d == 2) return prefix | ((1u << shift) - 1u);
    }
    return prefix;
}

template <bool FIRST, bool FINAL>
__global__ void __launch_bounds__(T, 2) topk_level_kernel(const __grid_constant__ Level p) {
    constexpr int E = FIRST ? E0 : E1;
    __shared__ uint32_t hist[2048];
    __shared__ uint32_t red[T / 32 + 4];
    __shared__ int cnt;
    __shared__ uint32_t wkey[FINAL ? TF_TOPK_MAX_K : 1], wcol[FINAL ? TF_TOPK_MAX_K : 1];
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();

    const int64_t row = blockIdx.x / p.nch;
    const int chunk = (int)(blockIdx.x - row * p.nch);
    const int t = threadIdx.x;
    uint32_t key[E], cidx[FIRST ? 1 : E];
    int64_t c0, m;
    if (FIRST) {
        int64_t len = p.n;
        if (p.len) {
            len = p.len[row];
            len = len < 0 ? 0 : (len > p.n ? p.n : len);
        }
        c0 = (int64_t)chunk * TF_TOPK_BLOCK;
        m = len - c0;
        const float *src = p.logits + row * p.ld + c0;
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {
            const int64_t b = 4 * (int64_t)(q * T + t);
            uint32_t u[4];
            if (b + 4 <= m) {
                const float4 v = __ldcs(reinterpret_cast<const float4 *>(src + b));
                u[0] = __float_as_uint(v.x);
                u[1] = __float_as_uint(v.y);
                u[2] = __float_as_uint(v.z);
                u[3] = __float_as_uint(v.w);
#pragma unroll
                for (int c = 0; c < 4; ++c) key[4 * q + c] = ord_key(u[c]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) key[4 * q + c] = b + c < m ? ord_key(__float_as_uint(src[b + c])) : 0u;
            }
        }
    } else {
        c0 = (int64_t)chunk * TF_TOPK_MERGE;
        m = p.cin_row - c0;
        const uint2 *src = p.cin + row * p.cin_row + c0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int64_t i = (int64_t)e * T + t;
            uint2 v = make_uint2(0u, kPad);
            if (i < m) v = __ldcs(src + i);
            key[e] = v.x;
            cidx[e] = v.y;
        }
    }
    // the column of entry e (kPad for a filler)
    auto col = [&](int e) -> uint32_t {
        if (FIRST) {
            const int64_t i = 4 * (int64_t)((e >> 2) * T + t) + (e & 3);
            return i < m ? (uint32_t)(c0 + i) : kPad;
        } else {
            return cidx[FIRST ? 0 : e];
        }
    };

    if (t == 0) cnt = 0;
    uint32_t lo, rem;
    bool all;
    key_select<E>(key, (uint32_t)p.k, hist, red, lo, rem, all);
    const uint32_t chi = all ? kPad : col_select<E>(key, col, lo, rem, hist, red);

    // compact the winners that are real keys; fillers make up the rest
    uint2 *dst = FINAL ? nullptr : p.cout + ((int64_t)row * p.nch + chunk) * p.k;
    const int lane = t & 31;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const uint32_t c = col(e);
        const bool take = c != kPad && (key[e] > lo || (key[e] == lo && c <= chi));
        const unsigned bal = __ballot_sync(0xffffffffu, take);
        int base = 0;
        if (lane == 0 && bal) base = atomicAdd(&cnt, __popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        const int o = base + __popc(bal & ((1u << lane) - 1u));
        if (take && o < p.k) {
            if (FINAL) {
                wkey[o] = key[e];
                wcol[o] = c;
            } else {
                dst[o] = make_uint2(key[e], c);
            }
        }
    }
    __syncthreads();
    const int have = cnt < p.k ? cnt : p.k;
    if (!FINAL) {
        for (int o = have + t; o < p.k; o += T) dst[o] = make_uint2(0u, kPad);
        return;
    }
    int kp = 1;
    while (kp < p.k) kp <<= 1;
    for (int o = have + t; o < kp; o += T) {
        wkey[o] = 0u;
        wcol[o] = kPad;
    }
    __syncthreads();
    // bitonic sort, best first: a larger key, then a smaller column (fillers last)
    for (int size = 2; size <= kp; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = t; i < kp; i += T) {
                const int j = i ^ stride;
                if (j > i) {
                    const uint32_t ka = wkey[i], kb = wkey[j], ca = wcol[i], cb = wcol[j];
                    const bool a_first = ka > kb || (ka == kb && ca < cb);
                    if (((i & size) == 0) != a_first) {
                        wkey[i] = kb;
                        wkey[j] = ka;
                        wcol[i] = cb;
                        wcol[j] = ca;
                    }
                }
            }
            __syncthreads();
        }
    const float *lrow = p.logits + row * p.ld;
    for (int i = t; i < p.k; i += T) {
        const uint32_t c = wcol[i], kk = wkey[i];
        int32_t oc = -1;
        float ov = -INFINITY;
        if (c != kPad) {
            oc = (int32_t)c;
            ov = kk != 0u ? __uint_as_float(key_bits(kk)) : lrow[c];  // a NaN keeps its own bits
        }
        p.out_idx[row * p.k + i] = oc;
        p.out_val[row * p.k + i] = ov;
    }
}

struct Plan {
    int64_t n0;     // first-level blocks a row
    int64_t n1;     // second-level blocks a row (0: the second level is the last)
};

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline Plan plan_of(int64_t n, int k) {
    Plan pl;
    pl.n0 = n > TF_TOPK_BLOCK ? cdiv(n, TF_TOPK_BLOCK) : 1;
    pl.n1 = 0;
    if (pl.n0 > 1) {
        const int64_t c = cdiv(pl.n0 * k, TF_TOPK_MERGE);
        pl.n1 = c > 1 ? c : 0;
    }
    return pl;
}

}  // namespace topk
}  // namespace tf

using namespace tf;
using namespace tf::topk;

extern "C" size_t tf_topk_workspace_bytes(int64_t rows, int64_t n, int32_t k) {
    if (rows <= 0 || n < 0 || k < 1 || k > TF_TOPK_MAX_K) return 0;
    const Plan pl = plan_of(n, k);
    if (pl.n0 == 1) return 0;
    return (size_t)rows * (size_t)(pl.n0 + pl.n1) * (size_t)k * sizeof(uint2);
}

extern "C" int tf_topk_blocked(const float *d_logits, int64_t rows, int64_t n, int64_t ld, const int32_t *d_len,
                               int32_t k, int32_t *d_idx, float *d_val, void *d_ws, size_t ws_bytes, void *stream) {
    if (rows < 0 || n < 0 || ld < n || k < 1 || k > TF_TOPK_MAX_K) return TF_E_ARG;
    if (rows == 0) return TF_OK;
    if (!d_logits || !d_idx || !d_val) return TF_E_ARG;
    if ((reinterpret_cast<uintptr_t>(d_logits) & 15u) || (ld & 3)) return TF_E_ARG;
    if (n > INT32_MAX) return TF_E_UNSUPPORTED;
    const size_t need = tf_topk_workspace_bytes(rows, n, k);
    if (need && (!d_ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(d_ws) & 15u))) return TF_E_NOMEM;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const Plan pl = plan_of(n, k);
    uint2 *A = static_cast<uint2 *>(d_ws);
    uint2 *B = A ? A + (size_t)rows * pl.n0 * k : nullptr;

    Level p = {};
    p.logits = d_logits;
    p.ld = ld;
    p.n = n;
    p.len = d_len;
    p.k = k;
    p.out_idx = d_idx;
    p.out_val = d_val;
    auto go = [&](auto kernel, int64_t nch) -> int {
        p.nch = (int32_t)nch;
        const int64_t blocks = rows * nch;
        if (blocks > INT32_MAX) return TF_E_UNSUPPORTED;
        const cudaError_t e = launch_pdl(kernel, dim3((unsigned)blocks), dim3(T), 0, st, p);
        launch_counter()++;
        return e == cudaSuccess ? TF_OK : TF_E_CUDA;
    };
    if (pl.n0 == 1) return go(topk_level_kernel<true, true>, 1);
    p.cout = A;
    int rc = go(topk_level_kernel<true, false>, pl.n0);
    if (rc != TF_OK) return rc;
    int64_t cur = pl.n0 * k;
    uint2 *in = A, *spare = B;
    for (;;) {
        const int64_t nch = cdiv(cur, TF_TOPK_MERGE);
        p.cin = in;
        p.cin_row = cur;
        if (nch == 1) return go(topk_level_kernel<false, true>, 1);
        p.cout = spare;
        rc = go(topk_level_kernel<false, false>, nch);
        if (rc != TF_OK) return rc;
        cur = nch * k;
        std::swap(in, spare);
    }
}
