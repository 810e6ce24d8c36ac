// Blocked top-k with an exact merge ("Running CHUNKED_PREFILL_SIZE above 1024 without the
// long-prompt memory problem", section 2.3): every block of a row keeps its top-k, the top-k of
// the candidates is the row's top-k.  Order: the IEEE total order of fp32 (a NaN below every
// number), larger first, ties by the smaller column.
//
// One CTA a block.  The block's keys live in registers (32 a thread for logits, 16 key/column
// pairs a thread for candidates), mapped to unsigned integers that compare like the values
// (merge blocks rescaled onto the whole range first).  One histogram of the top 11 bits finds
// the bin of the k-th key; the keys at or above it go to a shared list, where the select goes
// on with digits of 11 and 10 bits (stopping at the first digit whose bin is needed whole),
// and the keys equal to the k-th are ranked by counting their smaller columns (a radix pass
// over columns when there are many).  A block whose list overflows selects over the block
// again from global memory.  The winners are compacted with one shared atomic a warp; the last
// level sorts them (a bitonic network: registers, warp shuffles, then shared memory) and writes
// columns and values.
#include <cstdint>
#include <mutex>

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

// fp32 bits -> an unsigned key with the same order (the IEEE total order); every NaN -> 1,
// below -inf (whose key is 0x007FFFFF).  Key 0 marks a filler.
__device__ __forceinline__ uint32_t ord_key(uint32_t u) {
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 1u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The same map without the NaN rule (two instructions); equal to ord_key on every non-NaN.
// A NaN lands in bins 0-3 or 2044-2047 of the first digit, with the infinities.
__device__ __forceinline__ uint32_t ord_fast(uint32_t u) {
    return u ^ (uint32_t(int32_t(u) >> 31) | 0x80000000u);
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

// Digits of the radix select: 0 = bits 31..21 (the shared first pass), 1 = bits 20..10,
// 2 = bits 9..0.
__device__ __forceinline__ int dshift(int d) { return d == 0 ? 21 : (d == 1 ? 10 : 0); }
__device__ __forceinline__ int dbins(int d) { return d == 2 ? 1024 : 2048; }

// An order-preserving rescale of a merge block's real keys onto the whole 32-bit range
// (fillers stay 0): k -> (k - kmin + 1) << sh.  Merge candidates all sit near the top of the
// order, so without it most of them would share a first digit and its histogram counter.
// Identity for the first level (kmin 1, sh 0).
struct Scale {
    uint32_t kmin = 1;
    int sh = 0;
    __device__ __forceinline__ uint32_t fwd(uint32_t k) const { return k ? (k - kmin + 1u) << sh : 0u; }
    __device__ __forceinline__ uint32_t back(uint32_t k) const { return k ? (k >> sh) + kmin - 1u : 0u; }
};

// An entry set the selects can walk: the block re-read from global memory (each thread its
// own entries, as first loaded), or the shared list.
template <int E, bool FIRST>
struct Glob {
    const float *src;   // FIRST: the block's logits
    const uint2 *csrc;  // otherwise: the block's candidates
    uint32_t base;      // FIRST: column of the thread's entry 0
    int64_t m;          // entries of the block in play
    Scale sc;           // otherwise: the rescale of the keys in registers
    __device__ __forceinline__ uint32_t col(int e) const {
        if (FIRST) return base + 4u * (uint32_t)((e >> 2) * T) + (uint32_t)(e & 3);
        const int64_t i = (int64_t)e * T + threadIdx.x;
        return i < m ? csrc[i].y : kPad;
    }
    __device__ __forceinline__ uint32_t key(int e) const {
        if (FIRST) {
            const int64_t i = 4 * (int64_t)((e >> 2) * T + threadIdx.x) + (e & 3);
            return i < m ? ord_key(__float_as_uint(src[i])) : 0u;
        }
        const int64_t i = (int64_t)e * T + threadIdx.x;
        return i < m ? sc.fwd(csrc[i].x) : 0u;
    }
    template <class F>
    __device__ __forceinline__ void each(F f) const {  // f(valid, key, e): uniform over the CTA
#pragma unroll 4
        for (int e = 0; e < E; ++e) f(true, key(e), e);
    }
};
struct List {
    const uint32_t *key, *col_;
    int n;
    __device__ __forceinline__ uint32_t col(int i) const { return col_[i]; }
    template <class F>
    __device__ __forceinline__ void each(F f) const {
        for (int b = 0; b < n; b += T) {
            const int i = b + (int)threadIdx.x;
            const bool v = i < n;
            f(v, v ? key[i] : 0u, i);
        }
    }
};

// Digits d0..2 of the select among the entries whose key matches `prefix` on `pmask`; `rem` of
// them are wanted (1 <= rem <= their count).  Result: every key > lo is taken, and of the keys
// == lo either all (all) or the `rem` with the smallest columns.
template <class Set>
__device__ __forceinline__ void key_select(const Set &s, int d0, uint32_t prefix, uint32_t pmask, uint32_t rem,
                                           uint32_t *hist, uint32_t *red, uint32_t &lo, uint32_t &rem_out,
                                           bool &all) {
#pragma unroll 1
    for (int d = d0; d < 3; ++d) {
        const int shift = dshift(d), nb = dbins(d);
        for (int i = threadIdx.x; i < nb; i += T) hist[i] = 0;
        __syncthreads();
        s.each([&](bool v, uint32_t k, int) {
            if (v && (k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & (nb - 1)], 1u);
        });
        __syncthreads();
        const Bin r = find_bin<true>(hist, nb, rem, red);
        prefix |= r.bin << shift;
        pmask |= uint32_t(nb - 1) << shift;
        rem -= r.before;
        if (r.count == rem || d == 2) {
            lo = prefix;
            all = r.count == rem;
            rem_out = rem;
            return;
        }
    }
}

// Of the entries with key == lo, the `want` with the smallest columns: those with column <=
// the returned bound (columns are distinct among real keys).
template <class Set>
__device__ __forceinline__ uint32_t col_select(const Set &s, uint32_t lo, uint32_t want, uint32_t *hist,
                                               uint32_t *red) {
    uint32_t prefix = 0, pmask = 0, rem = want;
#pragma unroll 1
    for (int d = 0; d < 3; ++d) {
        const int shift = dshift(d), nb = dbins(d);
        for (int i = threadIdx.x; i < nb; i += T) hist[i] = 0;
        __syncthreads();
        s.each([&](bool v, uint32_t k, int e) {
            if (v && k == lo) {
                const uint32_t c = s.col(e);
                if ((c & pmask) == prefix) atomicAdd(&hist[(c >> shift) & (nb - 1)], 1u);
            }
        });
        __syncthreads();
        const Bin r = find_bin<false>(hist, nb, rem, red);
        prefix |= r.bin << shift;
        pmask |= uint32_t(nb - 1) << shift;
        rem -= r.before;
        if (r.count == rem || d == 2) return prefix | ((1u << shift) - 1u);
    }
    return prefix;
}

// Append the lanes' (key, column) where `take`, one shared atomic a warp: to og (global pairs)
// if given, else to okey (if given) and ocol.  All lanes call it.
__device__ __forceinline__ void append(bool take, uint32_t k, uint32_t c, int *counter, int cap, uint32_t *okey,
                                       uint32_t *ocol, uint2 *og) {
    const unsigned bal = __ballot_sync(0xffffffffu, take);
    if (!bal) return;
    const int lane = threadIdx.x & 31;
    int base = 0;
    if (lane == 0) base = atomicAdd(counter, __popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    const int o = base + __popc(bal & ((1u << lane) - 1u));
    if (take && o < cap) {
        if (og) {
            og[o] = make_uint2(k, c);
        } else {
            if (okey) okey[o] = k;
            ocol[o] = c;
        }
    }
}

constexpr int kCap = 4096;      // entries of the shared list
constexpr int kRankTies = 256;  // up to this many tied keys are ranked by counting
constexpr size_t kSmemBase = (2048 + 32) * 4 + 2 * (kCap + 4) * 4;
constexpr size_t kSmemFinal = kSmemBase + 2 * TF_TOPK_MAX_K * 4;


__device__ __forceinline__ bool ranks_first(uint32_t ka, uint32_t ca, uint32_t kb, uint32_t cb) {
    return ka > kb || (ka == kb && ca < cb);
}

// Bitonic sort of T*V (key, column) pairs, best first; element i = t*V + j sits in thread t,
// slot j.  Strides below V swap in registers, strides below 32*V through warp shuffles, the
// rest through shared memory, alternating between two buffers (x0 first, then x1; each a key
// and a column array of T*V words) so that one barrier a stage suffices: a buffer is written
// again only after the barrier of the stage that used the other.  Nothing may read x0 when
// the sort starts.
template <int V>
__device__ __forceinline__ void sort_best_first(uint32_t (&k)[V], uint32_t (&c)[V], uint32_t *x0k, uint32_t *x0c,
                                                uint32_t *x1k, uint32_t *x1c) {
    bool second = false;
    constexpr int N = T * V;
    const int t = threadIdx.x;
    // fully unrolled: every stage's masks are constants
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride < V) {
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    const int pj = j ^ stride;
                    if (pj > j) {
                        const bool up = ((t * V + j) & size) == 0;
                        if (up != ranks_first(k[j], c[j], k[pj], c[pj])) {
                            const uint32_t tk = k[j], tc = c[j];
                            k[j] = k[pj];
                            c[j] = c[pj];
                            k[pj] = tk;
                            c[pj] = tc;
                        }
                    }
                }
                continue;
            }
            uint32_t ok[V], oc[V];
            if (stride < 32 * V) {
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    ok[j] = __shfl_xor_sync(0xffffffffu, k[j], stride / V);
                    oc[j] = __shfl_xor_sync(0xffffffffu, c[j], stride / V);
                }
            } else {
                uint32_t *xk = second ? x1k : x0k, *xc = second ? x1c : x0c;
                second = !second;
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    xk[t * V + j] = k[j];
                    xc[t * V + j] = c[j];
                }
                __syncthreads();
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    ok[j] = xk[(t * V + j) ^ stride];
                    oc[j] = xc[(t * V + j) ^ stride];
                }
            }
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int i = t * V + j;
                const bool up = (i & size) == 0, lower = (i & stride) == 0;
                const bool mine = ranks_first(k[j], c[j], ok[j], oc[j]);
                if ((lower == up) != mine) {
                    k[j] = ok[j];
                    c[j] = oc[j];
                }
            }
        }
    }
}

// The last level: sort the `have` winners in wkey / wcol (fillers after them) and write the
// columns and values of the first k.  spare: 2 * TF_TOPK_MAX_K words nobody reads any more.
template <int V>
__device__ __forceinline__ void finish(const Level &p, int64_t row, int have, uint32_t *wkey, uint32_t *wcol,
                                       uint32_t *spare) {
    const int t = threadIdx.x;
    uint32_t k[V], c[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int i = t * V + j;
        k[j] = i < have ? wkey[i] : 0u;
        c[j] = i < have ? wcol[i] : kPad;
    }
    sort_best_first<V>(k, c, spare, spare + TF_TOPK_MAX_K, wkey, wcol);
    const float *lrow = p.logits + row * p.ld;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int i = t * V + j;
        if (i < p.k) {
            int32_t oc = -1;
            float ov = -INFINITY;
            if (k[j] != 0u) {
                oc = (int32_t)c[j];
                ov = k[j] != 1u ? __uint_as_float(key_bits(k[j])) : lrow[c[j]];  // a NaN keeps its own bits
            }
            p.out_idx[row * p.k + i] = oc;
            p.out_val[row * p.k + i] = ov;
        }
    }
}

// Select the top-k of one block whose keys (and, past the first level, columns) are in
// registers, and write them: candidates to p.cout, or (last level) sorted columns and values.
// c0: the block's first entry; m: its entries in play; fast: keys mapped by ord_fast.
template <bool FIRST, bool FINAL>
__device__ __forceinline__ void select_block(const Level &p, int64_t row, int chunk,
                                             uint32_t (&key)[FIRST ? E0 : E1],
                                             const uint32_t (&cidx)[FIRST ? 1 : E1], int64_t c0, int64_t m,
                                             bool fast, uint32_t *sm) {
    constexpr int E = FIRST ? E0 : E1;
    uint32_t *hist = sm;                 // [2048]
    uint32_t *red = sm + 2048;           // [T/32 + 4], then three counters
    int *cnt = reinterpret_cast<int *>(red + T / 32 + 4);
    int *lcnt = cnt + 1;
    int *tcnt = cnt + 2;
    uint32_t *lkey = sm + 2048 + 32;     // [kCap + 1]
    uint32_t *lcol = lkey + kCap + 4;    // [kCap + 1]
    uint32_t *wkey = lcol + kCap + 4;    // FINAL: [TF_TOPK_MAX_K]
    uint32_t *wcol = wkey + TF_TOPK_MAX_K;
    const int t = threadIdx.x;
    Scale sc;
    if (!FIRST) {
        // the real keys' range, then the rescale (hist holds the warps' partial results)
        uint32_t lo_k = 0xFFFFFFFFu, hi_k = 0u;
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (key[e]) {
                lo_k = min(lo_k, key[e]);
                hi_k = max(hi_k, key[e]);
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lo_k = min(lo_k, __shfl_xor_sync(0xffffffffu, lo_k, o));
            hi_k = max(hi_k, __shfl_xor_sync(0xffffffffu, hi_k, o));
        }
        if ((t & 31) == 0) {
            hist[t >> 5] = lo_k;
            hist[T / 32 + (t >> 5)] = hi_k;
        }
        __syncthreads();
#pragma unroll
        for (int w = 0; w < T / 32; ++w) {
            lo_k = min(lo_k, hist[w]);
            hi_k = max(hi_k, hist[T / 32 + w]);
        }
        __syncthreads();
        if (lo_k <= hi_k) {
            sc.kmin = lo_k;
            sc.sh = __clz(hi_k - lo_k + 1u);
#pragma unroll
            for (int e = 0; e < E; ++e) key[e] = sc.fwd(key[e]);
        }
    }
    Glob<E, FIRST> glob{FIRST ? p.logits + row * p.ld + c0 : nullptr,
                        FIRST ? nullptr : p.cin + row * p.cin_row + c0, (uint32_t)(c0 + 4 * t), m};
    glob.sc = sc;
    uint2 *dst = FINAL ? nullptr : p.cout + ((int64_t)row * p.nch + chunk) * p.k;
    uint32_t *okey = FINAL ? wkey : nullptr, *ocol = FINAL ? wcol : nullptr;

    // first digit over every entry (fillers fall in bin 0)
    for (int i = t; i < 2048; i += T) hist[i] = 0;
    if (t == 0) {
        *cnt = 0;
        *lcnt = 0;
        *tcnt = 0;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) atomicAdd(&hist[key[e] >> 21], 1u);
    __syncthreads();
    if (fast && (hist[0] | hist[1] | hist[2] | hist[3] | hist[2044] | hist[2045] | hist[2046] | hist[2047])) {
        // an infinity or a NaN: apply the NaN rule and count again
        __syncthreads();
        for (int i = t; i < 2048; i += T) hist[i] = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) key[e] = ord_key(key_bits(key[e]));
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) atomicAdd(&hist[key[e] >> 21], 1u);
        __syncthreads();
    }
    const Bin b0 = find_bin<true>(hist, 2048, (uint32_t)p.k, red);
    const uint32_t need = (uint32_t)p.k - b0.before;  // wanted from bin b0; every key above is taken
    const uint32_t lo0 = b0.bin << 21;
    const uint32_t floor = lo0 > 1u ? lo0 : 1u;        // the real keys in bin b0 or above

    // the keys in bin b0 or above go to the shared list: a count a thread, a scan a warp, one
    // atomic a warp, then predicated stores (slot kCap takes whatever does not fit)
    {
        int mine = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) mine += key[e] >= floor ? 1 : 0;
        const int lane = t & 31;
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int wbase = 0;
        if (lane == 31 && incl) wbase = atomicAdd(lcnt, incl);
        int o = __shfl_sync(0xffffffffu, wbase, 31) + incl - mine;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (key[e] >= floor) {
                const int at = o < kCap ? o : kCap;
                lkey[at] = key[e];
                lcol[at] = FIRST ? glob.base + 4u * (uint32_t)((e >> 2) * T) + (uint32_t)(e & 3) : cidx[FIRST ? 0 : e];
                ++o;
            }
        }
    }
    __syncthreads();
    const int nl = *lcnt;
    const uint32_t nbin = (uint32_t)nl - b0.before;   // real keys in bin b0
    const uint32_t want = need < nbin ? need : nbin;

    if (nl <= kCap) {
        const List list{lkey, lcol, nl};
        uint32_t lo = floor, rem = want;
        bool all = true;
        if (want < nbin) key_select(list, 1, lo0, 0x7FFu << 21, want, hist, red, lo, rem, all);
        int nt = 0;
        if (!all) {
            // the keys equal to lo: their columns side by side (in the histogram's room)
            list.each([&](bool v, uint32_t k, int i) {
                append(v && k == lo, 0u, v ? lcol[i] : 0u, tcnt, 2048, nullptr, hist, nullptr);
            });
            __syncthreads();
            nt = *tcnt;
        }
        if (all || nt <= kRankTies) {
            // a tie is taken when fewer than rem tied columns are smaller than its own
            list.each([&](bool v, uint32_t k, int i) {
                bool take = v && k > lo;
                if (v && k == lo) {
                    if (all) {
                        take = true;
                    } else {
                        const uint32_t c = lcol[i];
                        uint32_t below = 0;
                        for (int j = 0; j < nt; ++j) below += hist[j] < c ? 1u : 0u;
                        take = below < rem;
                    }
                }
                append(take, sc.back(k), v ? lcol[i] : 0u, cnt, p.k, okey, ocol, dst);
            });
        } else {
            __syncthreads();
            const uint32_t chi = col_select(list, lo, rem, hist, red);
            list.each([&](bool v, uint32_t k, int i) {
                const uint32_t c = v ? lcol[i] : 0u;
                append(v && (k > lo || (k == lo && c <= chi)), sc.back(k), c, cnt, p.k, okey, ocol, dst);
            });
        }
    } else {
        // too many keys share the first digit: select over the block again, from global memory
        uint32_t lo = floor, rem = want;
        bool all = true;
        if (want < nbin) key_select(glob, 1, lo0, 0x7FFu << 21, want, hist, red, lo, rem, all);
        if (lo == 0u) lo = 1u;
        const uint32_t chi = all ? 0xFFFFFFFFu : col_select(glob, lo, rem, hist, red);
#pragma unroll 4
        for (int e = 0; e < E; ++e) {
            const uint32_t k = glob.key(e);
            const bool cand = k >= floor && k >= lo;
            const uint32_t c = cand ? glob.col(e) : 0u;
            append(cand && (k > lo || c <= chi), sc.back(k), c, cnt, p.k, okey, ocol, dst);
        }
    }
    __syncthreads();
    const int have = *cnt < p.k ? *cnt : p.k;
    if (!FINAL) {
        for (int o = have + t; o < p.k; o += T) dst[o] = make_uint2(0u, kPad);
        return;
    }
    uint32_t *spare = lkey;  // the list is done with (lkey and lcol: 2 * (kCap + 4) words)
    if (p.k <= T)
        finish<1>(p, row, have, wkey, wcol, spare);
    else if (p.k <= 2 * T)
        finish<2>(p, row, have, wkey, wcol, spare);
    else
        finish<4>(p, row, have, wkey, wcol, spare);
}

template <bool FIRST, bool FINAL>
__global__ void __launch_bounds__(T, 2) topk_level_kernel(const __grid_constant__ Level p) {
    constexpr int E = FIRST ? E0 : E1;
    extern __shared__ __align__(16) uint32_t sm[];
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    const int t = threadIdx.x;
    uint32_t key[E], cidx[FIRST ? 1 : E];

    const int64_t row = blockIdx.x / p.nch;
    const int chunk = (int)(blockIdx.x - row * p.nch);
    int64_t c0, m;
    bool fast = false;  // keys mapped by ord_fast (a NaN not yet sent to 1)
    if (FIRST) {
        int64_t len = p.n;
        if (p.len) {
            len = p.len[row];
            len = len < 0 ? 0 : (len > p.n ? p.n : len);
        }
        c0 = (int64_t)chunk * TF_TOPK_BLOCK;
        m = len - c0;
        const float *src = p.logits + row * p.ld + c0;
        if (m >= TF_TOPK_BLOCK) {
            // a whole block: every load in flight before the first is used
            float4 v[E / 4];
#pragma unroll
            for (int q = 0; q < E / 4; ++q) v[q] = __ldcs(reinterpret_cast<const float4 *>(src) + q * T + t);
#pragma unroll
            for (int q = 0; q < E / 4; ++q) {
                key[4 * q + 0] = ord_fast(__float_as_uint(v[q].x));
                key[4 * q + 1] = ord_fast(__float_as_uint(v[q].y));
                key[4 * q + 2] = ord_fast(__float_as_uint(v[q].z));
                key[4 * q + 3] = ord_fast(__float_as_uint(v[q].w));
            }
            fast = true;
        } else if (m > 0) {
            // a ragged block: whole quads again (a quad that starts below m lies inside the
            // row's ld), quads past the end re-read quad 0; entries at or past m are fillers
            float4 v[E / 4];
#pragma unroll
            for (int q = 0; q < E / 4; ++q) {
                const int64_t b = 4 * (int64_t)(q * T + t);
                v[q] = __ldcs(reinterpret_cast<const float4 *>(src + (b < m ? b : 0)));
            }
#pragma unroll
            for (int q = 0; q < E / 4; ++q) {
                const int64_t b = 4 * (int64_t)(q * T + t);
                const uint32_t u[4] = {__float_as_uint(v[q].x), __float_as_uint(v[q].y), __float_as_uint(v[q].z),
                                       __float_as_uint(v[q].w)};
#pragma unroll
                for (int c = 0; c < 4; ++c) key[4 * q + c] = b + c < m ? ord_key(u[c]) : 0u;
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) key[e] = 0u;
        }
    } else {
        c0 = (int64_t)chunk * TF_TOPK_MERGE;
        m = p.cin_row - c0;
        const uint2 *src = p.cin + row * p.cin_row + c0;
        if (m >= TF_TOPK_MERGE) {
            uint2 v[E];
#pragma unroll
            for (int e = 0; e < E; ++e) v[e] = __ldcs(src + e * T + t);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                key[e] = v[e].x;
                cidx[e] = v[e].y;
            }
        } else {
            // a short block: every load issued (entries past m re-read entry 0), then masked
            uint2 v[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int64_t i = (int64_t)e * T + t;
                v[e] = __ldcs(src + (i < m ? i : 0));
            }
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const bool in = (int64_t)e * T + t < m;
                key[e] = in ? v[e].x : 0u;
                cidx[e] = in ? v[e].y : kPad;
            }
        }
    }
    select_block<FIRST, FINAL>(p, row, chunk, key, cidx, c0, m, fast, sm);
}

struct Plan {
    int64_t n0;     // first-level blocks a row
    int64_t n1;     // second-level blocks a row (0: the second level is the last)
};

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline size_t smem_of(void (*k)(Level)) {
    if (k == topk_level_kernel<true, true> || k == topk_level_kernel<false, true>) return kSmemFinal;
    return kSmemBase;
}

// Opt every instance in to its dynamic shared memory, once.
inline bool attributes_set() {
    static std::once_flag once;
    static bool ok = false;
    std::call_once(once, [] {
        ok = cudaFuncSetAttribute(topk_level_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemFinal) == cudaSuccess &&
             cudaFuncSetAttribute(topk_level_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemFinal) == cudaSuccess &&
             cudaFuncSetAttribute(topk_level_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemBase) == cudaSuccess &&
             cudaFuncSetAttribute(topk_level_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemBase) == cudaSuccess;
    });
    return ok;
}

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
    if (n > INT32_MAX || rows > INT32_MAX) return TF_E_UNSUPPORTED;
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
    if (!attributes_set()) return TF_E_CUDA;
    auto go = [&](auto kernel, int64_t nch) -> int {
        p.nch = (int32_t)nch;
        const int64_t blocks = rows * nch;
        if (blocks > INT32_MAX) return TF_E_UNSUPPORTED;
        const cudaError_t e = launch_pdl(kernel, dim3((unsigned)blocks), dim3(T), smem_of(kernel), st, p);
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
