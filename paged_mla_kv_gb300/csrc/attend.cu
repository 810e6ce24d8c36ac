// Absorbed-query attention over a paged latent cache (decode with 1-2 causal MTP
// rows, and prefill chunks), for sm_103a.
//
// What is computed (issue #1313, step 2 decode bullet: every head's absorbed query
// against one shared latent; issue #1142 "What stays as it is": the same key chunks
// merged in the same order whatever the pages):
//   out[s,r,h,:] = softmax_j(scale * q[s,r,h,:] . K_j) . C_j,  j <= len[s]-R+r
// with K_j = (latent C_j, rope Kr_j), 576 wide, and the value the 512-wide latent.
//
// Work (one persistent CTA an SM): a CTA walks segments, each one column group (up to 64
// (row, head) columns) of one stream over a run of its key tiles; how the tiles are dealt out
// (RANGES, UNITS, SPLITS, SPARSE) is described at the Params below.  Keys stream through
// 64-row tiles: 9 boxes of [64 keys x 64 values] bf16 (8 latent + 1 rope), loaded by TMA with
// 128-byte swizzle from the tile's pool page into a ring of 10 latent box-pair slots and 3 rope
// slots (2.5 tiles in flight).  A tile lands in two halves (rope box and pairs 0-1; pairs 2-3),
// and QK^T starts on the first while the second, whose slots free last, is still on its way.
// Listed rows on BF16 pages are copied row by row with cp.async by four loader warps into the
// same swizzled boxes.  The queries' latent values 0-255 sit in TMEM as the A operand
// of QK^T; only their last four latent boxes and the rope box stay in shared memory, which is
// what pays for the deeper ring.  The same shared-memory tile feeds both contractions on the
// 5th-generation tensor cores:
//   S   = Q . K^T     tcgen05.mma M=64 (the columns), N=64 keys, K=576, A from TMEM (values
//                     0-255) or shared memory (the rest), the tile K-major; S in TMEM (2 buffers)
//   O^T += V^T . P^T  tcgen05.mma M=128 latent values x 4, N = columns rounded up to 16,
//                     K=64 keys, the tile read MN-major as V^T, P (bf16, written into the tile's
//                     rope slot once QK^T has read it) K-major; O^T accumulates in TMEM (4 x 64 columns)
// Softmax is online in fp32 registers, each of four warps reading one TMEM lane quadrant
// (two rows and 16 of their keys a thread), with a lazily moved reference maximum: O^T is
// rescaled only when a tile's maximum passes the reference by more than 2^8, by a separate
// warp group.  A segment that is its whole unit writes bf16 output directly; a unit cut into
// several segments writes fp32 partials (unnormalised O, running maximum, sum) that a
// combine kernel merges in key order.
//
// Warp roles (352 threads; 480 on FP8 pages and for listed rows): warps 0-3 rescale O^T when
// asked and run the epilogue (one TMEM lane quadrant each); warps 4-7 softmax, and at each
// segment start write the segment's queries into TMEM; warp 8 the TMA producer; warp 9 the TMEM
// allocation and the QK^T issuer; warp 10 the PV issuer; on FP8 pages warps 11-14 expand each
// tile's codes to bf16 in shared memory, for listed rows on BF16 pages they copy the rows.  The MMA issuers walk their issue loops as whole warps with one elected lane
// issuing, in rolled loops: on this GPU both kept MMA issue markedly faster than a lone lane
// running unrolled issue code.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <memory>
#include <mutex>
#include <numeric>

#include "ptx.cuh"
#include "tf_internal.h"

namespace tf {

namespace attn {

constexpr int BK = 64;                          // keys a tile (N of the QK^T MMA: an MMA costs
                                                // about 49 cycles at N = 64 whether M is 64 or 128)
constexpr int NCOL = 64;                        // (row, head) columns a CTA
constexpr int NBOX = 9;                         // 64-wide boxes of a 576-wide row
constexpr int BOX_BYTES = BK * 128;             // [64 rows][64 bf16], 128B swizzle
constexpr int PAIR_BYTES = 2 * BOX_BYTES;       // latent boxes 2j and 2j+1 of a tile, side by side
constexpr int QBOX_BYTES = NCOL * 128;          // [64 columns][64 bf16]
// The queries: latent values 0-255 (boxes 0-3) sit in TMEM as the A operand of QK^T, written
// by the softmax warps at each segment start; latent boxes 4-7 and the rope box stay in shared
// memory (TMA).  Moving 32 KB of queries out of shared memory is what deepens the key ring; the
// rest of TMEM holds O^T and two S buffers, so QK^T of the next tile never waits for the
// softmax to read S out.
constexpr int Q_TMEM_BOXES = 4;
constexpr int Q_SMEM_BOXES = NBOX - Q_TMEM_BOXES;   // [latent 4 .. 7 | rope]
// The key ring: a tile is its rope box (in a rope slot) and four latent box pairs (in pair
// slots).  Pair slots are taken in order, four a tile (2.5 tiles in flight); a rope slot a tile
// (3 in flight).  Once QK^T has read a tile's rope box, the slot holds the tile's P for PV, so
// P is triple-buffered and the softmax never waits for the previous PV.
constexpr int NPAIR = 10;
constexpr int NROPE = 3;
constexpr int SMEM_Q = 0;
constexpr int SMEM_ROPE = SMEM_Q + Q_SMEM_BOXES * QBOX_BYTES;   // 40,960
constexpr int SMEM_PAIR = SMEM_ROPE + NROPE * BOX_BYTES;          // 65,536
constexpr int SMEM_CTRL = SMEM_PAIR + NPAIR * PAIR_BYTES;         // 229,376
constexpr float TAU = 8.0f;                     // lazy-rescale threshold, log2 units
constexpr int TMEM_COLS = 512;
constexpr int TMEM_O = 0;                       // O^T M-tile j at 64 j (j < 4)
constexpr int TMEM_S = 256;                     // S buffers at 256 and 320 (64 columns each)
constexpr int TMEM_Q = 384;                     // queries' latent values 0-255: column c holds values 2c, 2c+1
static_assert(TMEM_Q + Q_TMEM_BOXES * 32 == TMEM_COLS, "the queries fill TMEM's last columns");
constexpr int THREADS = 352;
// FP8 pages: four more warps (11-14) expand each tile's E4M3 codes into its BF16 boxes in place.
// The codes land by TMA, unswizzled, in the tile's pair slots 2-3 (the room of BF16 boxes 4-7):
// dense tiles as 8 boxes of 64 rows x 64 bytes (codes 64b.. of row r at pair slot 2 + b/4, byte
// 4 KB (b%4) + 64 r), gathered tiles as 2 blocks of 64 rows x 256 bytes (codes 256q.. of row r at
// pair slot 2 + q, byte 256 r; a quarter of the gathers).  BF16 box b (codes 64b..64b+63) is
// written in order, one pair slot a round, so each write covers only codes already read (the
// last round, boxes 6-7, reads all its rows first).
constexpr int THREADS_F8 = THREADS + 128;
constexpr int F8_THREADS = THREADS_F8 - THREADS;   // two threads a tile row
// Listed rows on BF16 pages: warps 11-14 copy each tile's rows with cp.async, 16 rows a warp
// (on this GPU 16-byte copies from four warps gather random 1 KB rows about twice as fast as
// TMA gather4 issued by one warp).
constexpr int LOAD_THREADS = 128;
template <int MODE, bool FP8>
constexpr int kernel_threads() { return FP8 || MODE == 3 ? THREADS + 128 : THREADS; }
constexpr int F8_BOX_BYTES = BK * 64;            // dense: [64 rows][64 codes]
constexpr int F8_BLK = 256;                      // gathered: codes a box row (the unswizzled maximum)
constexpr int F8_BLK_BYTES = BK * F8_BLK;        // [64 rows][256 codes] = 16 KB
constexpr int F8_NBLK = kLat / F8_BLK;           // 2
static_assert(4 * F8_BOX_BYTES == PAIR_BYTES && F8_BLK_BYTES == PAIR_BYTES, "a pair slot holds 4 code boxes or a block");
constexpr int MIN_TILES = 4;                    // fewest key tiles a CTA is given
constexpr int SPLIT_UNIT = 256;                 // batch-invariant split sizes are multiples of this
static_assert(SPLIT_UNIT % BK == 0, "splits must be tile-aligned");
constexpr int MAX_CTAS = 240;                   // CTAs a launch (one a SM); sizes the workspace
constexpr uint32_t IDESC_QK = ptx::idesc_bf16_f32(64, BK, false, false);

// Ring positions of global tile gt (the CTA's tiles counted across its segments): pair j sits in
// slot (4 gt + j) mod NPAIR for the ((4 gt + j) / NPAIR)-th time, the rope box in slot gt mod NROPE
// for the (gt / NROPE)-th time.  A slot's full and empty barriers complete once a use, so a wait
// for use u has parity u & 1.
__device__ __forceinline__ int pair_slot(int gt, int j) { return (4 * gt + j) % NPAIR; }
__device__ __forceinline__ uint32_t pair_use(int gt, int j) { return (uint32_t)((4 * gt + j) / NPAIR); }
__device__ __forceinline__ int rope_slot(int gt) { return gt % NROPE; }
__device__ __forceinline__ uint32_t rope_use(int gt) { return (uint32_t)(gt / NROPE); }
// Shared-memory offset of key box b (0-7 latent, 8 rope) of global tile gt.
__device__ __forceinline__ int box_off(int gt, int b) {
    return b == 8 ? SMEM_ROPE + rope_slot(gt) * BOX_BYTES : SMEM_PAIR + pair_slot(gt, b >> 1) * PAIR_BYTES + (b & 1) * BOX_BYTES;
}

// FP8: the tile's 64 row scales land (a bulk copy or the producer's stores) in the last 256
// bytes of its pair slot 1.  The expansion warps read them before the first round, and pair
// slot 1 is not written before the second.
__device__ __forceinline__ int scales_off(int gt) { return SMEM_PAIR + pair_slot(gt, 1) * PAIR_BYTES + PAIR_BYTES - BK * 4; }

struct Ctrl {
    uint64_t f8_full[NROPE];           // FP8: the tile's codes, scales and rope box landed
    uint64_t tile_half[NROPE];         // the tile's rope box and latent pairs 0-1 landed (FP8:
                                       // expanded); by rope slot
    uint64_t tile_full[NROPE];         // its latent pairs 2-3 landed (FP8: expanded)
    uint64_t rope_empty[NROPE];        // PV of the slot's tile is done (its rope box and P are free)
    uint64_t pair_empty[NPAIR];        // PV M-tile of the pair is done
    uint64_t p_full[NROPE];            // P of the slot's tile written and O^T rescaled for it
    uint64_t corr_req[NROPE];          // the tile's softmax statistics posted for the rescale warps
    uint64_t s_full[2], s_free[2];     // S buffer computed / read out of TMEM
    uint64_t q_full, q_tmem_full, q_free, stats_full, stats_free, drain;
    uint32_t tmem_base;
    int abort;
    int flag[NROPE];
    float alpha[NROPE][NCOL];
    float row_inv_l[2][NCOL];          // by segment parity
};
constexpr int SMEM_TOTAL = SMEM_CTRL + (int)sizeof(Ctrl) + 1024;
static_assert(SMEM_TOTAL <= 232448, "shared memory budget");

// How the work is dealt out to CTAs (one resident CTA a SM):
//  - RANGES (few column groups: decode, MTP rows).  The key tiles of the streams are
//    numbered stream by stream and cut into contiguous, near-equal ranges, so every
//    SM gets the same number of key tiles whatever the mix of lengths.  Each range is
//    taken by `rep` = groups CTAs side by side, one column group each, so the groups
//    of a stream read the same tiles at the same time.  A (stream, group) unit cut by
//    a range boundary leaves partials that a combine pass merges, in key order.
//  - UNITS (many column groups: a prefill chunk).  The units, stream-major, each only as
//    many key tiles as its last column sees, are numbered tile by tile and cut into equal
//    ranges of CTAs, like RANGES with one CTA a range: every SM gets the same work, where
//    whole units dealt round robin leave a tail round on some SMs only.  A cut inside a
//    long unit falls on an eighth of it, so the CTAs read at a few key positions in step
//    (the others' tiles come from L2).  A cut unit leaves partials, merged as in RANGES.
//  - SPLITS (a pool made with TF_POOL_BATCH_INVARIANT).  Each stream's keys are cut
//    into splits whose bounds depend on that stream's length alone, one CTA a
//    (split, group) item, and the partials are merged in split order, so a stream's
//    result has the same bits whatever else is in the batch.
//  - SPARSE (tf_paged_mla_attend_sparse).  RANGES over the tiles of each stream's list
//    of rows; the key tiles are gathered row by row (TMA gather4) through the table.
enum { MODE_RANGES = 0, MODE_UNITS = 1, MODE_SPLITS = 2, MODE_SPARSE = 3 };

// One entry per stream, in the caller's order.
struct StreamPlan {
    int64_t len;
    int64_t toff;     // RANGES: first numbered key tile of the stream
    int32_t nt;       // key tiles of the stream
    int32_t split;    // SPLITS: keys a split (a multiple of SPLIT_UNIT); SPARSE: the stream's rows
    int32_t nsplit;   // SPLITS: splits of each column group
    int32_t item0;    // SPLITS: first item of the stream (items are numbered in launch order)
    int32_t slot0;    // SPLITS: first workspace slot of the stream
    int32_t pad;
};

struct Params {
    CUtensorMap tm_lat;   // 4D {512, 512 rows, pages, caches}, box {64, 64, 1, 1}
    CUtensorMap tm_rope;  // 4D {64, 512 rows, pages, caches}, box {64, 64, 1, 1}
    CUtensorMap tm_q;     // 2D {576, S*R*H}, box {64, 64}
    CUtensorMap tm_lat_rows;    // SPARSE: 2D {512, pool rows}, 1,024-byte rows (576 a page), box {64, 1}
    CUtensorMap tm_rope_rows;   // SPARSE: 2D {64, pool rows}, 128-byte rows (4,608 a page), box {64, 1}
    const int32_t *idx;         // SPARSE: [S][max_idx] row numbers of each stream's listed keys
    int32_t max_idx;
    const int32_t *pt;
    const __nv_bfloat16 *q;     // [S*R*H][576]: the TMEM part of each column group is read from here
    __nv_bfloat16 *out;
    float *lse;
    float *ws_o;          // [slots][64][512]
    float *ws_ml;         // [slots][64][2]
    DevErr *err;
    const char *pool_base;  // FP8: the pool (row scales are read from each page)
    int64_t total;        // RANGES: numbered key tiles; UNITS: units
    float scale_log2;
    int32_t cache, max_pages, num_pages, S, R, H, ncols, groups, windowed;
    int32_t mode;
    int32_t nranges;      // RANGES: ranges of the numbering
    int32_t rep;          // RANGES: CTAs a range (the column groups)
    int64_t rb[MAX_CTAS + 1];        // RANGES: range i is tiles [rb[i], rb[i+1]); UNITS: positions
    StreamPlan st[TF_MAX_STREAMS];
    int16_t order[TF_MAX_STREAMS];   // SPLITS: launch order (streams with longer splits first)
};

// UNITS: keys unit (stream of `len` keys, column group g) reads, up to the last key its last
// column sees (the R rows are the stream's last R positions; column c is row c / H).  len >= R.
__host__ __device__ __forceinline__ int64_t unit_keys(int64_t len, int R, int H, int ncols, int g) {
    const int64_t clast = (int64_t)g * NCOL + NCOL - 1 < ncols ? (int64_t)g * NCOL + NCOL - 1 : (int64_t)ncols - 1;
    return len - R + clast / H + 1;
}
// UNITS: a position of the numbering, (unit, tile within it), as one ordered integer
__host__ __device__ __forceinline__ int64_t unit_pos(int64_t u, int64_t t) { return (u << 32) | t; }

// The range that holds numbered tile x (UNITS: position x).
__device__ __forceinline__ int range_of(const Params &p, int64_t x) {
    int lo = 0, hi = p.nranges - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.rb[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// A CTA's range, cut at unit boundaries: each piece (a segment) attends one column
// group of one stream over a contiguous run of key tiles.
struct Seg {
    int s, g, nt;
    int slot;          // workspace slot of a partial result; -1: the segment is its whole unit
    int64_t kb, ke;    // keys [kb, ke)
    int64_t len;
};

__device__ __forceinline__ Seg seg_at(const Params &p, int64_t x, int64_t x0, int64_t x1) {
    int lo = 0, hi = p.S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.st[mid].toff <= x) lo = mid; else hi = mid - 1;
    }
    Seg q;
    q.s = lo;
    const int64_t toff = p.st[lo].toff, len = p.st[lo].len;
    const int nt = p.st[lo].nt;
    const int64_t u = x - toff;
    (void)u;
    q.g = (int)blockIdx.x % p.rep;
    const int64_t ub = toff, ue = ub + nt;
    const int64_t tin = x - ub;
    const int64_t e = ue < x1 ? ue : x1;
    q.nt = (int)(e - x);
    q.kb = tin * BK;
    q.ke = min(len, (tin + q.nt) * BK);
    q.len = len;
    // a CTA holds at most two partial segments: its first and its last
    q.slot = (x == ub && e == ue) ? -1 : 2 * (int)blockIdx.x + (x == x0 ? 0 : 1);
    return q;
}

// This CTA's segments, in order, for every mode.
// The kernel is compiled once per mode, so each instance carries only its own plan.
template <int MODE>
struct SegIter {
    int64_t x, x0, x1;
    int k;
    __device__ __forceinline__ explicit SegIter(const Params &p) : x(0), x0(0), x1(0), k(0) {
        if (MODE == MODE_RANGES || MODE == MODE_SPARSE || MODE == MODE_UNITS) {
            const int range = (int)blockIdx.x / p.rep;
            x0 = p.rb[range];
            x1 = p.rb[range + 1];
            x = x0;
        }
    }
    // after next() returned a segment: is it this CTA's last?
    __device__ __forceinline__ bool last(const Params &p) const {
        if (MODE == MODE_RANGES || MODE == MODE_SPARSE || MODE == MODE_UNITS) return x >= x1;
        return true;
    }
    __device__ __forceinline__ bool next(const Params &p, Seg &q) {
        if (MODE == MODE_RANGES || MODE == MODE_SPARSE) {
            if (x >= x1) return false;
            q = seg_at(p, x, x0, x1);
            x += q.nt;
            return true;
        }
        if (MODE == MODE_UNITS) {
            // the rest of unit u from tile t: up to the range's end or the unit's last tile
            if (x >= x1) return false;
            const int64_t u = x >> 32, t = x & 0xffffffffll;
            q.s = (int)(u / p.groups);
            q.g = (int)(u - (int64_t)q.s * p.groups);
            q.len = p.st[q.s].len;
            const int64_t keys = unit_keys(q.len, p.R, p.H, p.ncols, q.g);
            const int64_t nt = (keys + BK - 1) / BK;
            const int64_t te = (x1 >> 32) == u ? (x1 & 0xffffffffll) : nt;
            q.nt = (int)(te - t);
            q.kb = t * BK;
            q.ke = min(keys, te * BK);
            q.slot = (t == 0 && te == nt) ? -1 : 2 * (int)blockIdx.x + (k == 0 ? 0 : 1);
            ++k;
            x = te == nt ? unit_pos(u + 1, 0) : unit_pos(u, te);
            return true;
        }
        // SPLITS: one item a CTA
        if (k++ > 0) return false;
        const int item = (int)blockIdx.x;
        int lo = 0, hi = p.S - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.st[p.order[mid]].item0 <= item) lo = mid; else hi = mid - 1;
        }
        q.s = p.order[lo];
        const StreamPlan &sp = p.st[q.s];
        // items of a stream run split-major, so the column groups of one split read the
        // same key tiles at about the same time
        const int local = item - sp.item0;
        const int j = local / p.groups;
        q.g = local - j * p.groups;
        q.len = sp.len;
        q.kb = (int64_t)j * sp.split;
        q.ke = min(sp.len, q.kb + (int64_t)sp.split);
        q.nt = (int)((q.ke - q.kb + BK - 1) / BK);
        q.slot = sp.nsplit > 1 ? sp.slot0 + q.g * sp.nsplit + j : -1;
        return true;
    }
};

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *tm, uint64_t *bar, int c0, int c1, int c2,
                                            int c3, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(ptx::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(ptx::smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "l"(policy)
        : "memory");
}

#define ALLW(x) __all_sync(0xffffffffu, (x))

// Barrier phases: a parity wait only tells the current phase from the one before it, so a
// barrier may be neither two phases ahead of a waiter nor two phases short of the phase it
// waits for.  Slot barriers count the slot's uses; s_full / s_free the CTA's tiles (gt);
// q_full, q_tmem_full, q_free, stats_full, stats_free its segments (si).  What keeps each
// within one phase:
//  - p_full and corr_req are indexed like the rope slots: the softmax of tile gt + 3 needs the
//    tile to land in rope slot gt mod 3, which needs PV(gt), which needs p_full(gt) (from the
//    softmax and the rescale warps) to have been consumed;
//  - "PV of tile gt is done" is rope_empty of its slot: the rescale warps (before moving O^T)
//    and the epilogue wait on it, and tile gt having landed means its slot's previous use is
//    released, so the barrier is never two phases short;
//  - the softmax waits stats_free (the epilogue read the previous segment's statistics) before
//    posting a segment's stats_full, so stats_full is never two phases ahead of the epilogue;
//  - the first PV of a segment waits p_full, which the rescale warps post only after their
//    epilogue of the previous segment has read the accumulator.

template <int MODE, bool FP8 = false>
__global__ void __launch_bounds__(kernel_threads<MODE, FP8>(), 1) mla_attend_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // listed rows on BF16 pages arrive by the loader warps' cp.async copies
    constexpr bool CP_ROWS = MODE == MODE_SPARSE && !FP8;
    Ctrl &c = *reinterpret_cast<Ctrl *>(smem + SMEM_CTRL);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_launch_dependents();

    // every per-launch scalar the roles use, copied out of the parameter block once
    const float scale_log2 = p.scale_log2;
    const int R_ = p.R, H_ = p.H, ncols_all = p.ncols, ngroups = p.groups;
    const int max_pages = p.max_pages, num_pages = p.num_pages, cache = p.cache;
    const bool windowed = p.windowed != 0;
    const int32_t *const pt = p.pt;
    __nv_bfloat16 *const outp = p.out;
    float *const lsep = p.lse;
    float *const ws_o = p.ws_o;
    float *const ws_ml = p.ws_ml;
    DevErr *const errp = p.err;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NROPE; ++i) {
            // BF16: the TMA warp's one arrival with the tile's bytes; FP8: one arrival a pair the
            // expansion warps finish
            ptx::mbar_init(&c.tile_full[i], FP8 ? 2 : CP_ROWS ? LOAD_THREADS : 1);
            ptx::mbar_init(&c.tile_half[i], FP8 ? 2 : CP_ROWS ? LOAD_THREADS : 1);
            ptx::mbar_init(&c.rope_empty[i], 1);
            ptx::mbar_init(&c.p_full[i], 5);       // four softmax warps and the rescale warps
            ptx::mbar_init(&c.corr_req[i], 4);
            // FP8: the codes' copies (and, for listed rows, the producer's scale stores)
            if (FP8) ptx::mbar_init(&c.f8_full[i], MODE == MODE_SPARSE ? 2 : 1);
            c.flag[i] = 0;
        }
        for (int i = 0; i < NPAIR; ++i) {
            ptx::mbar_init(&c.pair_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&c.s_full[i], 1);
            ptx::mbar_init(&c.s_free[i], 4);
        }
        ptx::mbar_init(&c.q_full, 1);
        ptx::mbar_init(&c.q_tmem_full, 4);
        ptx::mbar_init(&c.q_free, 1);
        ptx::mbar_init(&c.stats_full, 4);
        ptx::mbar_init(&c.stats_free, 4);
        ptx::mbar_init(&c.drain, 2);
        c.abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 9) {
        ptx::tmem_alloc(&c.tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = c.tmem_base;
    volatile int *abort = &c.abort;
    // on-chip setup done: from here on global memory (pool, tables, queries, outputs)
    ptx::griddep_wait();

    // A tile lands in two halves: QK^T starts on the rope box and latent pairs 0-1 while pairs
    // 2-3, whose slots the PV of the tile two back releases last, are still on their way (FP8:
    // still being expanded).  Two waits a tile, not one a pair: a wait costs about four MMAs.
    if (warp == 8) {
        // ================= TMA producer =================
        // Slot uses armed last (-1: never), so that no copy is left writing shared memory at exit.
        int armed_tile[NROPE], armed_f8[NROPE];
        for (int i = 0; i < NROPE; ++i) armed_tile[i] = armed_f8[i] = -1;
        int q_armed = -1;   // last segment whose queries were loaded
        bool stop = false;
        // wait until the tile's rope slot is released by PV of its previous tile (lane 0); BF16
        // pages then arm the tile's two landing barriers (rope box and pairs 0-1; pairs 2-3)
        auto take_rope = [&](int gt) -> bool {
            const int rs = rope_slot(gt);
            const uint32_t u = rope_use(gt);
            if (u > 0 && !ptx::mbar_wait(&c.rope_empty[rs], (u - 1) & 1, abort, errp, 1)) return false;
            if (!FP8) {
                ptx::mbar_arrive_expect_tx(&c.tile_half[rs], 5 * BOX_BYTES);
                ptx::mbar_arrive_expect_tx(&c.tile_full[rs], 4 * BOX_BYTES);
                armed_tile[rs] = (int)u;
            }
            return true;
        };
        auto free_pair = [&](int gt, int j) -> bool {
            const uint32_t u = pair_use(gt, j);
            return u == 0 || ptx::mbar_wait(&c.pair_empty[pair_slot(gt, j)], (u - 1) & 1, abort, errp, 1);
        };
        if constexpr (MODE == MODE_SPARSE) {
            // Gathered key tiles: list position k0 + 2l and + 1 belong to lane l; rows 4j..4j+3
            // of every box are one gather4 by lane j (< 16), from the table's page of each row.
            if (lane == 0) {
                ptx::prefetch_tmap(&p.tm_lat_rows);
                ptx::prefetch_tmap(&p.tm_rope_rows);
                ptx::prefetch_tmap(&p.tm_q);
            }
            const uint64_t pol_kv = ptx::policy_evict_first();
            const uint64_t pol_q = ptx::policy_evict_last();
            int gt = 0, si = 0;
            SegIter<MODE> it(p);
            Seg q;
            for (; !stop && it.next(p, q); ++si) {
                int okq = 1;
                if (lane == 0) {
                    if (si > 0 && !ptx::mbar_wait(&c.q_free, (si - 1) & 1, abort, errp, 15)) {
                        okq = 0;
                    } else {
                        ptx::mbar_arrive_expect_tx(&c.q_full, Q_SMEM_BOXES * QBOX_BYTES);
                        const int qrow = q.s * R_ * H_ + q.g * NCOL;
                        for (int b = 0; b < Q_SMEM_BOXES; ++b)
                            ptx::tma_load_2d(smem + SMEM_Q + b * QBOX_BYTES, &p.tm_q, &c.q_full,
                                             (Q_TMEM_BOXES + b) * 64, qrow, pol_q);
                    }
                }
                if (!__shfl_sync(0xffffffffu, okq, 0)) break;
                q_armed = si;
                if constexpr (CP_ROWS) continue;   // the loader warps copy the rows
                const int32_t *list = p.idx + (size_t)q.s * p.max_idx;
                const int rows = p.st[q.s].split;
                // list position k0 + 2 lane + h of tile tl2; past the list's end a listed row is
                // loaded again (the softmax masks it)
                auto list_at = [&](int tl2, int h) -> int {
                    const int64_t pos = q.kb + (int64_t)tl2 * BK + 2 * lane + h;
                    return __ldg(list + (pos < q.len ? pos : 0));
                };
                // the pool page of a listed row (-1 for a row outside the stream)
                auto page_of = [&](int r) -> int {
                    if (r < 0 || r >= rows) return -1;
                    const int lp = r >> 9;
                    return windowed ? q.s * max_pages + lp : __ldg(pt + (int64_t)q.s * max_pages + lp);
                };
                // the list entries run two tiles and their pages one tile ahead of the copies, so
                // these dependent loads overlap the waits for free slots instead of delaying each tile
                int rc[2], pc[2], rn[2], pn[2] = {0, 0}, rnn[2] = {0, 0};
#pragma unroll
                for (int h = 0; h < 2; ++h) rc[h] = list_at(0, h);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    pc[h] = page_of(rc[h]);
                    rn[h] = q.nt > 1 ? list_at(1, h) : 0;
                }
                for (int tl = 0; tl < q.nt; ++tl, ++gt) {
                    if (tl > 0) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            rc[h] = rn[h];
                            pc[h] = pn[h];
                            rn[h] = rnn[h];
                        }
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        pn[h] = tl + 1 < q.nt ? page_of(rn[h]) : 0;
                        rnn[h] = tl + 2 < q.nt ? list_at(tl + 2, h) : 0;
                    }
                    const int rs = rope_slot(gt);
                    int ylat[2], yrope[2], badv = 0;
                    const char *sc_addr[2] = {nullptr, nullptr};
                    bool bad = false;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int r = rc[h];
                        int pg = pc[h];
                        if (r < 0 || r >= rows) {
                            bad = true;
                            badv = r;
                            pg = 0;
                        } else if (pg < 0 || pg >= num_pages) {
                            bad = true;
                            badv = pg;
                            pg = 0;
                        }
                        const int base = cache * num_pages + pg;
                        // rows of the views: 1,024-byte latent rows (576 a page) and 128-byte rope
                        // rows (4,608 a page) on BF16 pages; 512-byte code rows (644 a page) and
                        // 128-byte rope rows (2,576 a page) on FP8 pages
                        constexpr int kLatRowsPerPage = FP8 ? (int)(kF8PageBytes / kLat) : (int)(kPageBytes / (kLat * 2));
                        constexpr int kRopeRowsPerPage = FP8 ? (int)(kF8PageBytes / (kRope * 2)) : (int)(kPageBytes / (kRope * 2));
                        ylat[h] = base * kLatRowsPerPage + (r & 511);
                        yrope[h] = base * kRopeRowsPerPage + (r & 511);
                        if (FP8) sc_addr[h] = p.pool_base + (size_t)base * kF8PageBytes + kF8ScaleOff + (size_t)(r & 511) * 4;
                    }
                    const unsigned badm = __ballot_sync(0xffffffffu, bad);
                    if (badm) {
                        const int v = __shfl_sync(0xffffffffu, badv, __ffs(badm) - 1);
                        if (lane == 0) {
                            ptx::record_error(errp, TF_E_DEVICE, v);
                            *abort = 1;
                        }
                        stop = true;
                        break;
                    }
                    const int jl = lane & 15;
                    const int la0 = __shfl_sync(0xffffffffu, ylat[0], 2 * jl), la1 = __shfl_sync(0xffffffffu, ylat[1], 2 * jl);
                    const int la2 = __shfl_sync(0xffffffffu, ylat[0], 2 * jl + 1),
                              la3 = __shfl_sync(0xffffffffu, ylat[1], 2 * jl + 1);
                    const int ro0 = __shfl_sync(0xffffffffu, yrope[0], 2 * jl), ro1 = __shfl_sync(0xffffffffu, yrope[1], 2 * jl);
                    const int ro2 = __shfl_sync(0xffffffffu, yrope[0], 2 * jl + 1),
                              ro3 = __shfl_sync(0xffffffffu, yrope[1], 2 * jl + 1);
                    if constexpr (FP8) {
                        // the tile's rope slot and all four pair slots must be free (the codes and
                        // their expansion cover the pairs)
                        int okw = 1;
                        if (lane == 0) {
                            okw = take_rope(gt);
                            for (int j = 0; okw && j < 4; ++j) okw = free_pair(gt, j);
                            if (okw) {
                                ptx::mbar_arrive_expect_tx(&c.f8_full[rs], F8_NBLK * F8_BLK_BYTES + BOX_BYTES);
                                armed_f8[rs] = (int)rope_use(gt);
                            }
                        }
                        if (!__shfl_sync(0xffffffffu, okw, 0)) {
                            stop = true;
                            break;
                        }
                        __syncwarp();
                        if (lane < 16) {
                            ptx::tma_gather4(smem + box_off(gt, 8) + lane * 512, &p.tm_rope_rows, &c.f8_full[rs], 0,
                                             ro0, ro1, ro2, ro3, pol_kv);
                            // rows 4j..4j+3 of code block qb: 4 x 256 bytes, unswizzled, in pair slot 2 + qb
                            for (int qb = 0; qb < F8_NBLK; ++qb)
                                ptx::tma_gather4(smem + SMEM_PAIR + pair_slot(gt, 2 + qb) * PAIR_BYTES + lane * 4 * F8_BLK,
                                                 &p.tm_lat_rows, &c.f8_full[rs], qb * F8_BLK, la0, la1, la2, la3,
                                                 pol_kv);
                        }
                        // the row scales: each lane its two listed rows; a second arrival
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            reinterpret_cast<float *>(smem + scales_off(gt))[2 * lane + h] =
                                __ldg(reinterpret_cast<const float *>(sc_addr[h]));
                        __threadfence_block();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(&c.f8_full[rs]);
                    } else {
                    // the rope box, then the latent pairs in order
                    for (int j = -1; j < 4; ++j) {
                        int okw = 1;
                        if (lane == 0) {
                            okw = j < 0 ? take_rope(gt) : free_pair(gt, j);
                        }
                        if (!__shfl_sync(0xffffffffu, okw, 0)) {
                            stop = true;
                            break;
                        }
                        if (lane < 16) {
                            uint64_t *bar = j < 2 ? &c.tile_half[rs] : &c.tile_full[rs];
                            if (j < 0) {
                                ptx::tma_gather4(smem + box_off(gt, 8) + lane * 512, &p.tm_rope_rows, bar, 0, ro0, ro1,
                                                 ro2, ro3, pol_kv);
                            } else {
                                for (int h = 0; h < 2; ++h)
                                    ptx::tma_gather4(smem + box_off(gt, 2 * j + h) + lane * 512, &p.tm_lat_rows, bar,
                                                     (2 * j + h) * 64, la0, la1, la2, la3, pol_kv);
                            }
                        }
                    }
                    }
                    if (stop) break;
                }
            }
        } else if (lane == 0) {
            ptx::prefetch_tmap(&p.tm_lat);
            ptx::prefetch_tmap(&p.tm_rope);
            ptx::prefetch_tmap(&p.tm_q);
            // a key tile read by one column group streams through L2; tiles that other
            // groups of the same stream read too are kept
            const uint64_t pol_kv = ngroups > 2 ? ptx::policy_evict_last() : ptx::policy_evict_first();
            const uint64_t pol_q = ptx::policy_evict_last();
            int gt = 0, si = 0;
            SegIter<MODE> it(p);
            Seg q;
            for (; !stop && it.next(p, q); ++si) {
                // the queries' shared-memory boxes are reloaded once the previous segment's QK^T has read them
                if (si > 0 && !ptx::mbar_wait(&c.q_free, (si - 1) & 1, abort, errp, 15)) break;
                ptx::mbar_arrive_expect_tx(&c.q_full, Q_SMEM_BOXES * QBOX_BYTES);
                const int qrow = q.s * R_ * H_ + q.g * NCOL;
                for (int b = 0; b < Q_SMEM_BOXES; ++b)
                    ptx::tma_load_2d(smem + SMEM_Q + b * QBOX_BYTES, &p.tm_q, &c.q_full, (Q_TMEM_BOXES + b) * 64, qrow,
                                     pol_q);
                q_armed = si;
                int cur_lp = -1, page = 0;
                for (int tl = 0; tl < q.nt; ++tl, ++gt) {
                    const int rs = rope_slot(gt);
                    const int64_t k0 = q.kb + (int64_t)tl * BK;
                    const int lp = (int)(k0 >> 9), row = (int)(k0 & 511);
                    if (lp != cur_lp) {
                        const int raw = windowed ? q.s * max_pages + lp : __ldg(pt + (int64_t)q.s * max_pages + lp);
                        cur_lp = lp;
                        if (raw < 0 || raw >= num_pages) {
                            ptx::record_error(errp, TF_E_DEVICE, raw);
                            *abort = 1;
                            stop = true;
                            break;
                        }
                        page = raw;
                    }
                    if constexpr (FP8) {
                        // the codes land in pair slots 2-3 and their expansion covers all four
                        // pairs: every slot of the tile must be free; the rope box lands as on BF16 pages
                        bool okw = take_rope(gt);
                        for (int j = 0; okw && j < 4; ++j) okw = free_pair(gt, j);
                        if (!okw) {
                            stop = true;
                            break;
                        }
                        ptx::mbar_arrive_expect_tx(&c.f8_full[rs], BOX_BYTES + 8 * F8_BOX_BYTES + BK * 4);
                        tma_load_4d(smem + box_off(gt, 8), &p.tm_rope, &c.f8_full[rs], 0, row, page, cache, pol_kv);
                        for (int b = 0; b < 8; ++b)
                            tma_load_4d(smem + SMEM_PAIR + pair_slot(gt, 2 + (b >> 2)) * PAIR_BYTES + (b & 3) * F8_BOX_BYTES,
                                        &p.tm_lat, &c.f8_full[rs], b * 64, row, page, cache, pol_kv);
                        ptx::bulk_g2s(smem + scales_off(gt),
                                      p.pool_base + ((size_t)cache * num_pages + page) * kF8PageBytes + kF8ScaleOff +
                                          (size_t)row * 4,
                                      BK * 4, &c.f8_full[rs]);
                        armed_f8[rs] = (int)rope_use(gt);
                    } else {
                        // the rope box first (QK^T starts on it), then the latent pairs in order
                        if (!take_rope(gt)) {
                            stop = true;
                            break;
                        }
                        tma_load_4d(smem + box_off(gt, 8), &p.tm_rope, &c.tile_half[rs], 0, row, page, cache, pol_kv);
#pragma unroll 1
                        for (int j = 0; j < 4; ++j) {
                            if (!free_pair(gt, j)) {
                                stop = true;
                                break;
                            }
                            uint64_t *bar = j < 2 ? &c.tile_half[rs] : &c.tile_full[rs];
                            for (int h = 0; h < 2; ++h)
                                tma_load_4d(smem + box_off(gt, 2 * j + h), &p.tm_lat, bar, (2 * j + h) * 64, row, page,
                                            cache, pol_kv);
                        }
                        if (stop) break;
                    }
                }
            }
        }
        // no copy may still be writing shared memory when the CTA exits
        if (lane == 0) {
            if (q_armed >= 0) ptx::mbar_wait(&c.q_full, q_armed & 1, abort, errp, 10, 1ll << 28);
            for (int i = 0; i < NROPE; ++i) {
                if (armed_tile[i] >= 0) {
                    ptx::mbar_wait(&c.tile_half[i], armed_tile[i] & 1, abort, errp, 11, 1ll << 28);
                    ptx::mbar_wait(&c.tile_full[i], armed_tile[i] & 1, abort, errp, 11, 1ll << 28);
                }
                if (armed_f8[i] >= 0) ptx::mbar_wait(&c.f8_full[i], armed_f8[i] & 1, abort, errp, 18, 1ll << 28);
            }
        }
        __syncwarp();
    } else if (warp == 9 || warp == 10) {
        // ================= MMA issuers =================
        // Warp 9 issues QK^T tile by tile as key boxes land; warp 10 issues PV as the softmax
        // publishes P.  Each accumulator gets its contributions in a fixed order, so timing
        // never changes a bit.
        const bool qk_role = warp == 9;
        const uint64_t q_desc0 = ptx::sdesc_sw128(ptx::smem_u32(smem + SMEM_Q), 16, 1024);
        const uint64_t kv_desc0 = ptx::sdesc_sw128(ptx::smem_u32(smem), 16, 1024);
        const uint64_t v_desc0 = ptx::sdesc_sw128(ptx::smem_u32(smem + SMEM_PAIR), BOX_BYTES, 1024);
        const uint64_t p_desc0 = ptx::sdesc_sw128(ptx::smem_u32(smem + SMEM_ROPE), 16, 1024);
        // QK^T of global tile tq (tile tl of segment q): S[64 columns][64 keys] (M = 64: rows
        // 16w..16w+15 in lanes 0-15 of TMEM quadrant w; buffer tq % 2).  Box order: rope (queries'
        // rope box in shared memory), latent pairs 0-1 (queries in TMEM), pairs 2-3 (shared memory).
        auto qk_tile = [&](int tq, int tl, const Seg &q) -> bool {
            const int rs = rope_slot(tq);
            // the tile's S buffer has been read out (by the softmax of tile tq - 2)
            if (tq >= 2 && !ptx::mbar_wait_warp(&c.s_free[tq & 1], ((tq - 2) >> 1) & 1, abort, errp, 4)) return false;
            const int64_t rem = q.len - (q.kb + (int64_t)tl * BK);
            // rows past the stream's end may hold NaN poison: zero them in latent boxes [b0, b1) and
            // the rope box, so that P = 0 times V stays 0 in the PV contraction
            auto zero_box = [&](int b) {
                const int valid = (int)rem;
                uint4 *bx = reinterpret_cast<uint4 *>(smem + box_off(tq, b));
                for (int k = lane; k < (BK - valid) * 8; k += 32) bx[valid * 8 + k] = make_uint4(0, 0, 0, 0);
            };
            auto zero_tail = [&](int b0, int b1, bool rope) {
                if (rem >= BK) return;
                if (rope) zero_box(8);
                for (int b = b0; b < b1; ++b) zero_box(b);
                ptx::fence_proxy_async_smem();
                __syncwarp();
            };
            const uint32_t d = tmem + TMEM_S + (tq & 1) * BK;
            // latent boxes [b0, b1): 0-3 with the queries' values from TMEM, 4-7 from shared memory;
            // a rolled loop keeps this warp's code small in the instruction cache
            auto latent = [&](int b0, int b1) {
                int ps = pair_slot(tq, b0 >> 1);
#pragma unroll 1
                for (int b = b0; b < b1; ++b) {
                    const uint64_t bd = kv_desc0 + (uint64_t)((SMEM_PAIR + ps * PAIR_BYTES + (b & 1) * BOX_BYTES) >> 4);
                    if (b < Q_TMEM_BOXES)
                        ptx::mma4_bf16_ts_warp(d, tmem + TMEM_Q + 32 * b, bd, IDESC_QK);
                    else
                        ptx::mma4_bf16_ss_warp(d, q_desc0 + (uint64_t)(((b - Q_TMEM_BOXES) * QBOX_BYTES) >> 4), bd,
                                               IDESC_QK, 0u);
                    if ((b & 1) && ++ps == NPAIR) ps = 0;
                }
            };
            // the tile's first half has landed (a wait costs about as long as four MMAs, so the
            // MMAs go out in runs of 20 and 16)
            if (!ptx::mbar_wait_warp(&c.tile_half[rs], rope_use(tq) & 1, abort, errp, 3)) return false;
            // rows copied by cp.async (generic proxy) become visible to the tensor cores' reads
            if (CP_ROWS) ptx::fence_proxy_async_smem();
            zero_tail(0, 4, true);
            // order the MMAs after the softmax's TMEM loads of S (s_free) and the queries' TMEM
            // stores (q_tmem_full, waited before a segment's first tile); the key boxes come by
            // TMA and need no such fence
            ptx::tc_fence_after();
            // the rope box (queries' rope box in shared memory) starts S, then the latent pairs
            ptx::mma4_bf16_ss_warp(d, q_desc0 + (uint64_t)(((Q_SMEM_BOXES - 1) * QBOX_BYTES) >> 4),
                                   kv_desc0 + (uint64_t)((SMEM_ROPE + rs * BOX_BYTES) >> 4), IDESC_QK, 1u);
            latent(0, 4);
            // the second half
            if (!ptx::mbar_wait_warp(&c.tile_full[rs], rope_use(tq) & 1, abort, errp, 3)) return false;
            if (CP_ROWS) ptx::fence_proxy_async_smem();
            zero_tail(4, 8, false);
            latent(4, 8);
            ptx::mma_commit_warp(&c.s_full[tq & 1]);
            if (tl == q.nt - 1) ptx::mma_commit_warp(&c.q_free);
            return true;
        };
        // PV of global tile tv (tile tl of segment q); each latent pair is released as soon as its
        // M-tile's MMAs finish, the rope slot (P) after the last; a segment's first tile starts
        // the accumulator
        auto pv_tile = [&](int tv, int tl, uint32_t idesc_pv) -> bool {
            const int rs = rope_slot(tv);
            if (!ptx::mbar_wait_warp(&c.p_full[rs], rope_use(tv) & 1, abort, errp, 5)) return false;
            ptx::tc_fence_after();
            {
                const uint64_t pd = p_desc0 + (uint64_t)((rs * BOX_BYTES) >> 4);
                const uint32_t acc0 = tl == 0 ? 0u : 1u;
#pragma unroll 1
                for (int jm = 0; jm < 4; ++jm) {
                    const int ps = pair_slot(tv, jm);
                    const uint64_t vd = v_desc0 + (uint64_t)((ps * PAIR_BYTES) >> 4);
                    // K = 64 keys in four steps: 16 keys of V^T (2 KB of the pair slot), 16 keys of P (32 bytes)
                    ptx::mma4_bf16_ss_step_warp(tmem + TMEM_O + jm * 64, vd, pd, idesc_pv, acc0, 2048 >> 4, 32 >> 4);
                    ptx::mma_commit_warp(&c.pair_empty[ps]);
                }
                ptx::mma_commit_warp(&c.rope_empty[rs]);
            }
            __syncwarp();
            return true;
        };
        bool ok = true;
        int gt = 0, si = 0;
        SegIter<MODE> it(p);
        Seg q;
        for (; ok && it.next(p, q); ++si) {
            const int ncols = min(NCOL, ncols_all - q.g * NCOL);
            const uint32_t idesc_pv = ptx::idesc_bf16_f32(128, (ncols + 15) & ~15, true, false);
            if (qk_role) {
                ok = ptx::mbar_wait_warp(&c.q_full, si & 1, abort, errp, 2) &&
                     ptx::mbar_wait_warp(&c.q_tmem_full, si & 1, abort, errp, 2);
                for (int tl = 0; ok && tl < q.nt; ++tl) ok = qk_tile(gt + tl, tl, q);
            } else {
                for (int tl = 0; ok && tl < q.nt; ++tl) ok = pv_tile(gt + tl, tl, idesc_pv);
            }
            gt += q.nt;
        }
        // drain: no MMA may still run when TMEM is freed
        if (lane == 0) {
            ptx::mma_commit(&c.drain);
            ptx::mbar_wait(&c.drain, 0, abort, errp, 6, 1ll << 29);
        }
        __syncwarp();
    } else if (CP_ROWS && warp >= 11) {
        // ================= listed-row loaders (warps 11-14): rows 16 lw .. 16 lw + 15 of each tile =================
        // A listed row is 1,024 bytes of latent values and 128 of rope: 64 + 8 copies of 16 bytes
        // into the 128-byte-swizzled boxes (chunk c of tile row r at r * 128 + 16 (c ^ (r mod 8))).
        // The rope box and latent boxes 0-3 (pairs 0-1) complete tile_half, boxes 4-7 tile_full;
        // each barrier counts one arrival a loader thread, made once its earlier copies are done.
        const int lw = warp - 11;
        const uint64_t pol_kv = ptx::policy_evict_first();
        bool stop = false;
        int gt = 0;
        SegIter<MODE> it(p);
        Seg q;
        // lane 0 waits until pair j of tile gt (j < 0: its rope slot) is free, for the whole warp
        auto slot_free = [&](int j) -> bool {
            int ok = 1;
            if (lane == 0) {
                const uint32_t u = j < 0 ? rope_use(gt) : pair_use(gt, j);
                uint64_t *bar = j < 0 ? &c.rope_empty[rope_slot(gt)] : &c.pair_empty[pair_slot(gt, j)];
                ok = u == 0 || ptx::mbar_wait(bar, (u - 1) & 1, abort, errp, 19);
            }
            return __shfl_sync(0xffffffffu, ok, 0) != 0;
        };
        while (!stop && it.next(p, q)) {
            const int32_t *list = p.idx + (size_t)q.s * p.max_idx;
            const int rows = p.st[q.s].split;
            for (int tl = 0; tl < q.nt; ++tl, ++gt) {
                const int rs = rope_slot(gt);
                // lane l < 16: tile row 16 lw + l, from its page (past the list's end a listed row
                // is copied again; the softmax masks it)
                const char *base = nullptr;   // the row's page
                int ri = 0, bad = 0, badv = 0;
                if (lane < 16) {
                    const int64_t pos = q.kb + (int64_t)tl * BK + 16 * lw + lane;
                    const int r = __ldg(list + (pos < q.len ? pos : 0));
                    if (r < 0 || r >= rows) {
                        bad = 1;
                        badv = r;
                    } else {
                        const int lp = r >> 9;
                        const int pg = windowed ? q.s * max_pages + lp : __ldg(pt + (int64_t)q.s * max_pages + lp);
                        if (pg < 0 || pg >= num_pages) {
                            bad = 1;
                            badv = pg;
                        } else {
                            base = p.pool_base + ((size_t)cache * num_pages + pg) * kPageBytes;
                            ri = r & 511;
                        }
                    }
                }
                const unsigned badm = __ballot_sync(0xffffffffu, bad);
                if (badm) {
                    const int v = __shfl_sync(0xffffffffu, badv, __ffs(badm) - 1);
                    if (lane == 0) {
                        ptx::record_error(errp, TF_E_DEVICE, v);
                        *abort = 1;
                    }
                    stop = true;
                    break;
                }
                // each row's latent and rope addresses, from the lane that looked it up: shuffled
                // once a tile, so a copy costs few instructions (this loop is issue-bound)
                const char *lat_src = base + (size_t)ri * (kLat * 2);
                const char *rope_src = base + kLatBlockBytes + (size_t)ri * (kRope * 2);
                const char *lat[16];
#pragma unroll
                for (int rr = 0; rr < 16; ++rr)
                    lat[rr] = reinterpret_cast<const char *>(__shfl_sync(0xffffffffu, (unsigned long long)lat_src, rr));
                // this lane's 16-byte chunk c = lane mod 8 of box lane / 8 (+ 4 in the second half):
                // row tr = 16 lw + rr sits at tr * 128 + 16 (c ^ (tr mod 8)), and tr mod 8 = rr mod 8
                const int c8 = lane & 7;
                // first half: the rope box (four rows an instruction) and latent values 0-255
                if (!slot_free(-1) || !slot_free(0) || !slot_free(1)) {
                    stop = true;
                    break;
                }
                {
                    uint8_t *dst = smem + box_off(gt, lane >> 3) + 16 * lw * 128;
#pragma unroll
                    for (int rr = 0; rr < 16; ++rr)
                        ptx::cp_async16(dst + rr * 128 + ((c8 ^ (rr & 7)) << 4), lat[rr] + lane * 16, pol_kv);
                    uint8_t *rdst = smem + box_off(gt, 8) + 16 * lw * 128;
#pragma unroll
                    for (int g4 = 0; g4 < 4; ++g4) {
                        const int rr = 4 * g4 + (lane >> 3);
                        const char *src = reinterpret_cast<const char *>(
                            __shfl_sync(0xffffffffu, (unsigned long long)rope_src, rr));
                        ptx::cp_async16(rdst + rr * 128 + ((c8 ^ (rr & 7)) << 4), src + c8 * 16, pol_kv);
                    }
                }
                ptx::cp_async_arrive(&c.tile_half[rs]);
                // second half: latent values 256-511 (pairs 2-3)
                if (!slot_free(2) || !slot_free(3)) {
                    stop = true;
                    break;
                }
                {
                    uint8_t *dst = smem + box_off(gt, 4 + (lane >> 3)) + 16 * lw * 128;
#pragma unroll
                    for (int rr = 0; rr < 16; ++rr)
                        ptx::cp_async16(dst + rr * 128 + ((c8 ^ (rr & 7)) << 4), lat[rr] + 512 + lane * 16, pol_kv);
                }
                ptx::cp_async_arrive(&c.tile_full[rs]);
            }
        }
        // no copy may still be writing shared memory when the CTA exits
        ptx::cp_async_wait_all();
        __syncwarp();
    } else if (FP8 && warp >= 11) {
        // ================= FP8 expansion (warps 11-14): half a tile row a thread =================
        // Box b's 64 codes of row r become bf16(code * scale_r), written 128B-swizzled into BF16
        // box b (16-byte chunk j of the row at j ^ (r & 7)); thread (r, hf) does codes 32hf..+31.
        // Each finished pair is one arrival on the tile's half barrier (pairs 0-1) or full barrier
        // (pairs 2-3), after a proxy fence.
        const int ft = (int)threadIdx.x - THREADS;
        const int r = ft >> 1, hf = ft & 1;
        bool ok = true;
        int gt = 0;
        SegIter<MODE> it(p);
        Seg q;
        while (ok && it.next(p, q)) {
            for (int tl = 0; tl < q.nt; ++tl, ++gt) {
                const int rs = rope_slot(gt);
                const bool landed = ptx::mbar_wait_warp(&c.f8_full[rs], rope_use(gt) & 1, abort, errp, 16);
                if (ptx::named_bar_or(2, F8_THREADS, !landed || *abort)) {
                    ok = false;
                    break;
                }
                const float sc = reinterpret_cast<const float *>(smem + scales_off(gt))[r];
                // one pair a round: {0,1}, {2,3}, {4,5}, {6,7}
#pragma unroll 1
                for (int b0 = 0; b0 < 8; b0 += 2) {
                    uint4 cv[2][2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int b = b0 + u;   // codes 64b.. of row r, in the dense or the gathered layout
                        const int off = SMEM_PAIR + pair_slot(gt, 2 + (b >> 2)) * PAIR_BYTES +
                                        (MODE == MODE_SPARSE ? r * F8_BLK + (b & 3) * 64 : (b & 3) * F8_BOX_BYTES + r * 64);
                        const uint4 *src = reinterpret_cast<const uint4 *>(smem + off + hf * 32);
                        cv[u][0] = src[0];
                        cv[u][1] = src[1];
                    }
                    uint32_t o[2][16];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const uint32_t w4[4] = {cv[u][k].x, cv[u][k].y, cv[u][k].z, cv[u][k].w};
#pragma unroll
                            for (int wi = 0; wi < 4; ++wi)
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
                                        (__nv_fp8x2_storage_t)((w4[wi] >> (16 * h)) & 0xFFFFu), __NV_E4M3);
                                    const float2 f = __half22float2(__half2(hr));
                                    o[u][k * 8 + wi * 2 + h] = ptx::pack_bf16x2(f.x * sc, f.y * sc);
                                }
                        }
                    // boxes 6-7 cover their own codes: every row read before any is overwritten
                    if (b0 == 6) ptx::named_bar(2, F8_THREADS);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        uint8_t *dst = smem + box_off(gt, b0 + u) + r * 128;
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int j = 4 * hf + jj;
                            *reinterpret_cast<uint4 *>(dst + ((j ^ (r & 7)) << 4)) =
                                make_uint4(o[u][4 * jj], o[u][4 * jj + 1], o[u][4 * jj + 2], o[u][4 * jj + 3]);
                        }
                    }
                    ptx::fence_proxy_async_smem();
                    ptx::named_bar(2, F8_THREADS);
                    if (ft == 0) ptx::mbar_arrive(b0 < 4 ? &c.tile_half[rs] : &c.tile_full[rs]);
                }
            }
        }
    } else if (warp >= 4) {
        // ================= softmax (warps 4-7: TMEM quadrant w holds S rows 16w..16w+15) =================
        // A 16x256b load gives thread t rows r0 = 16w + t/4 and r1 = r0 + 8, keys
        // 8j + 2(t%4) + {0, 1} for j < 8: a row's 64 keys are spread over 4 threads.
        const int q4 = warp & 3;
        const int r0 = 16 * q4 + (lane >> 2), r1 = r0 + 8;
        const int kq = 2 * (lane & 3);
        const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
        bool ok = true;
        int gt = 0, si = 0;
        SegIter<MODE> it(p);
        Seg q;
        for (; ok && it.next(p, q); ++si) {
            const int col0 = q.g * NCOL;
            const int ncols = ncols_all - col0;
            {
                // The segment's queries, latent values 0-255, into TMEM (A of QK^T): lane i < 16 of
                // this quadrant holds column 16 q4 + i.  Every QK^T of the previous segment has
                // completed: this warp has seen its last S.
                const int m = 16 * q4 + (lane & 15);
                const bool live = lane < 16 && m < ncols;
                const uint4 *src = reinterpret_cast<const uint4 *>(p.q + ((size_t)q.s * ncols_all + col0 + (live ? m : 0)) * kDk);
#pragma unroll 1
                for (int c2 = 0; c2 < Q_TMEM_BOXES; c2 += 2) {
                    uint32_t v[2][32];
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint4 x = live ? __ldg(src + (c2 + h) * 8 + i) : make_uint4(0, 0, 0, 0);
                            v[h][4 * i] = x.x;
                            v[h][4 * i + 1] = x.y;
                            v[h][4 * i + 2] = x.z;
                            v[h][4 * i + 3] = x.w;
                        }
                    ptx::tmem_st32(lane_base + TMEM_Q + 32 * c2, v[0]);
                    ptx::tmem_st32(lane_base + TMEM_Q + 32 * (c2 + 1), v[1]);
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&c.q_tmem_full);
            }
            const bool act0 = r0 < ncols, act1 = r1 < ncols;
            // last visible key of each row's column
            const int64_t pos0 = q.len - R_ + (act0 ? (col0 + r0) / H_ : 0);
            const int64_t pos1 = q.len - R_ + (act1 ? (col0 + r1) / H_ : 0);
            float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
            for (int tl = 0; tl < q.nt; ++tl) {
                const int t = gt + tl;
                const int rs = rope_slot(t);
                const int64_t k0 = q.kb + (int64_t)tl * BK;
                if (!ptx::mbar_wait_warp(&c.s_full[t & 1], (t >> 1) & 1, abort, errp, 7)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                uint32_t r[32];
                ptx::tmem_ld_16x256b_x8(lane_base + TMEM_S + (t & 1) * BK, r);
                ptx::tmem_ld_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&c.s_free[t & 1]);
                // keys outside a row's range become -inf; the maximum is taken before
                // scaling (the scale is positive) and the scale is folded into the
                // exponent's FFMA: p = 2^(s * scale*log2(e) - m_ref)
                const int64_t lim0 = (pos0 + 1 < q.ke ? pos0 + 1 : q.ke) - k0;
                const int64_t lim1 = (pos1 + 1 < q.ke ? pos1 + 1 : q.ke) - k0;
                const int nv0 = act0 ? (lim0 < 0 ? 0 : (lim0 > BK ? BK : (int)lim0)) : 0;
                const int nv1 = act1 ? (lim1 < 0 ? 0 : (lim1 > BK ? BK : (int)lim1)) : 0;
                float x0[16], x1[16];
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    x0[2 * j] = __uint_as_float(r[4 * j]);
                    x0[2 * j + 1] = __uint_as_float(r[4 * j + 1]);
                    x1[2 * j] = __uint_as_float(r[4 * j + 2]);
                    x1[2 * j + 1] = __uint_as_float(r[4 * j + 3]);
                }
                // only a range's or a stream's last tile (and causal rows) hold keys to mask
                if (!__all_sync(0xffffffffu, (nv0 == BK) & (nv1 == BK))) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int key = 8 * j + kq;
                        if (key >= nv0) x0[2 * j] = -INFINITY;
                        if (key + 1 >= nv0) x0[2 * j + 1] = -INFINITY;
                        if (key >= nv1) x1[2 * j] = -INFINITY;
                        if (key + 1 >= nv1) x1[2 * j + 1] = -INFINITY;
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    mx0 = fmaxf(mx0, fmaxf(x0[2 * j], x0[2 * j + 1]));
                    mx1 = fmaxf(mx1, fmaxf(x1[2 * j], x1[2 * j + 1]));
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mt0 = mx0 * scale_log2, mt1 = mx1 * scale_log2;
                float a0 = 1.f, a1 = 1.f;
                if (mt0 > m0 + TAU) {
                    a0 = (m0 == -INFINITY) ? 0.f : ptx::ex2(m0 - mt0);
                    m0 = mt0;
                    l0 *= a0;
                }
                if (mt1 > m1 + TAU) {
                    a1 = (m1 == -INFINITY) ? 0.f : ptx::ex2(m1 - mt1);
                    m1 = mt1;
                    l1 *= a1;
                }
                if ((lane & 3) == 0) {
                    c.alpha[rs][r0] = a0;
                    c.alpha[rs][r1] = a1;
                }
                if (__any_sync(0xffffffffu, (a0 != 1.f || a1 != 1.f) && tl > 0) && lane == 0) atomicOr(&c.flag[rs], 1);
                const float mr0 = (m0 == -INFINITY) ? 0.f : m0, mr1 = (m1 == -INFINITY) ? 0.f : m1;
                uint32_t pk0[8], pk1[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float e00 = ptx::ex2(fmaf(x0[2 * j], scale_log2, -mr0));
                    const float e01 = ptx::ex2(fmaf(x0[2 * j + 1], scale_log2, -mr0));
                    const float e10 = ptx::ex2(fmaf(x1[2 * j], scale_log2, -mr1));
                    const float e11 = ptx::ex2(fmaf(x1[2 * j + 1], scale_log2, -mr1));
                    l0 += e00 + e01;
                    l1 += e10 + e11;
                    pk0[j] = ptx::pack_bf16x2(e00, e01);
                    pk1[j] = ptx::pack_bf16x2(e10, e11);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&c.corr_req[rs]);
                // P rows as bf16, 128B-swizzled K-major, into the tile's rope slot (QK^T has read
                // the rope box: S is complete): keys 8j.. of row r in 16-byte chunk j ^ (r & 7)
                uint8_t *pb = smem + SMEM_ROPE + rs * BOX_BYTES;
                uint8_t *p0 = pb + r0 * 128 + 2 * kq;
                uint8_t *p1 = pb + r1 * 128 + 2 * kq;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    *reinterpret_cast<uint32_t *>(p0 + ((j ^ (r0 & 7)) << 4)) = pk0[j];
                    *reinterpret_cast<uint32_t *>(p1 + ((j ^ (r1 & 7)) << 4)) = pk1[j];
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&c.p_full[rs]);
            }
            if (!ok) break;
            // the row sums: each thread holds 16 of a row's keys a tile
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            // the epilogue of the previous segment must have read its statistics
            if (si > 0 && !ptx::mbar_wait_warp(&c.stats_free, (si - 1) & 1, abort, errp, 17)) {
                ok = false;
                break;
            }
            if ((lane & 3) == 0) {
                c.row_inv_l[si & 1][r0] = l0 > 0.f ? 1.f / l0 : 0.f;
                c.row_inv_l[si & 1][r1] = l1 > 0.f ? 1.f / l1 : 0.f;
                for (int h = 0; h < 2; ++h) {
                    const int rr = h ? r1 : r0;
                    const float m = h ? m1 : m0, l = h ? l1 : l0;
                    if (!(h ? act1 : act0)) continue;
                    if (q.slot < 0) {
                        if (lsep) lsep[(size_t)q.s * ncols_all + col0 + rr] = (m + log2f(l)) * 0.69314718055994531f;
                    } else {
                        ws_ml[((size_t)q.slot * NCOL + rr) * 2 + 0] = m;
                        ws_ml[((size_t)q.slot * NCOL + rr) * 2 + 1] = l;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&c.stats_full);
            gt += q.nt;
        }
    } else {
        // ================= rescale on request, then the epilogue (warps 0-3) =================
        const int q4 = warp;
        const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
        bool ok = true;
        int gt = 0, si = 0;
        SegIter<MODE> it(p);
        Seg q;
        for (; ok && it.next(p, q); ++si) {
            const int col0 = q.g * NCOL;
            const int ncols = min(NCOL, ncols_all - col0);
            const int npv = (ncols + 15) & ~15;
            for (int tl = 0; tl < q.nt; ++tl) {
                const int t = gt + tl;
                const int rs = rope_slot(t);
                if (!ptx::mbar_wait_warp(&c.corr_req[rs], rope_use(t) & 1, abort, errp, 12)) ok = false;
                const bool do_corr = ok && c.flag[rs] != 0;   // set only for tl > 0
                if (do_corr) {
                    // O^T holds every tile before t once PV(t - 1) is done
                    if (!ptx::mbar_wait_warp(&c.rope_empty[rope_slot(t - 1)], rope_use(t - 1) & 1, abort, errp, 13))
                        ok = false;
                    if (ok) {
                        ptx::tc_fence_after();
                        for (int jm = 0; jm < 4; ++jm)
                            for (int h2 = 0; h2 < npv; h2 += 32) {
                                uint32_t v[32];
                                const uint32_t a = lane_base + TMEM_O + jm * 64 + h2;
                                ptx::tmem_ld32(a, v);
                                ptx::tmem_ld_wait();
#pragma unroll
                                for (int k = 0; k < 32; ++k)
                                    v[k] = __float_as_uint(__uint_as_float(v[k]) * c.alpha[rs][h2 + k]);
                                ptx::tmem_st32(a, v);
                            }
                        ptx::tmem_st_wait();
                    }
                }
                // also orders the previous segment's epilogue reads of the accumulator
                // before the PV that starts it afresh
                ptx::tc_fence_before();
                if (ptx::named_bar_or(1, 128, !ok || *abort)) {
                    ok = false;
                    break;
                }
                if (threadIdx.x == 0) {
                    c.flag[rs] = 0;
                    ptx::mbar_arrive(&c.p_full[rs]);
                }
            }
            const int tlast = gt + q.nt - 1;
            if (ok && !*abort) {
                if (!ptx::mbar_wait_warp(&c.stats_full, si & 1, abort, errp, 14)) ok = false;
                if (ok && !ptx::mbar_wait_warp(&c.rope_empty[rope_slot(tlast)], rope_use(tlast) & 1, abort, errp, 9))
                    ok = false;
            }
            if (ptx::named_bar_or(1, 128, !ok || *abort)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const float *inv_l = c.row_inv_l[si & 1];
            if (q.slot >= 0 && it.last(p)) {
                // The CTA's last segment, cut: its fp32 partial (up to 128 KB: the columns PV
                // computed, in 32-column steps) goes out by one bulk copy from shared memory,
                // staged in the key ring, which no tile uses any more (the last PV is done and the
                // TMA warp loads nothing after it).  Every CTA ends with this write at about the
                // same time; one bulk copy a CTA moves it faster than 4,096 warp stores.
                float *stage = reinterpret_cast<float *>(smem + SMEM_PAIR);
                const int nst = (npv + 31) & ~31;
                for (int jm = 0; jm < 4; ++jm)
                    for (int h2 = 0; h2 < nst; h2 += 32) {
                        uint32_t v[32];
                        ptx::tmem_ld32(lane_base + TMEM_O + jm * 64 + h2, v);
                        ptx::tmem_ld_wait();
                        const int dim = jm * 128 + q4 * 32 + lane;
#pragma unroll
                        for (int k = 0; k < 32; ++k) stage[(h2 + k) * kLat + dim] = __uint_as_float(v[k]);
                    }
                ptx::fence_proxy_async_smem();
                ptx::named_bar(1, 128);
                if (threadIdx.x == 0) {
                    ptx::bulk_s2g(ws_o + (size_t)q.slot * NCOL * kLat, stage, nst * kLat * sizeof(float));
                    ptx::bulk_s2g_wait();
                }
            } else {
                for (int jm = 0; jm < 4; ++jm)
                    for (int h2 = 0; h2 < npv; h2 += 32) {
                        uint32_t v[32];
                        ptx::tmem_ld32(lane_base + TMEM_O + jm * 64 + h2, v);
                        ptx::tmem_ld_wait();
                        const int dim = jm * 128 + q4 * 32 + lane;
    #pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const int col = h2 + k;
                            if (col >= ncols) continue;
                            const float o = __uint_as_float(v[k]);
                            if (q.slot < 0) {
                                const size_t orow = (size_t)q.s * ncols_all + col0 + col;
                                outp[orow * kLat + dim] = __float2bfloat16_rn(o * inv_l[col]);
                            } else {
                                ws_o[((size_t)q.slot * NCOL + col) * kLat + dim] = o;
                            }
                        }
                    }
            }
            // the statistics are read: the softmax may post the next segment's
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&c.stats_free);
            gt += q.nt;
        }
    }

    // ---- teardown ----
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 9) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

// Merge a unit's partials (m_j, l_j, o_j), j in key order:
//   M = max_j m_j,  w_j = 2^(m_j - M),  out = sum_j w_j o_j / sum_j w_j l_j,
//   lse = (M + log2 sum_j w_j l_j) * ln 2.
// Lane l of a warp holds values 4 (l + 32 i) .. + 3 (i < 4) of one column.
//  - Few partials a unit (at most 8, the common case for listed rows, short batches and prefill
//    chunks): a block per (stream, column group, four columns), a warp a column, adding the
//    partials one after another in key order; the lanes first fetch the (m_j, l_j) pairs side
//    by side, 32 at a time.
//  - More partials (long streams cut by many ranges): a 256-thread block per (stream, column);
//    warp w adds
//    the partials j = w, w + 8, ... in key order and the eight warp sums are added in warp
//    order.
// Either way the order is fixed, so the result is the same on every call.  UNITS: blockIdx.y is
// a range bound, and a bound inside a unit that no earlier bound cuts stands for that unit.
constexpr int COMBINE_THREADS = 256;
constexpr int COMBINE_COLS = 4;         // columns a block of the warp-a-column form
constexpr int COMBINE_NARROW_MAX = 8;   // partials a unit that form takes

// The unit (stream s, group g) of a combine block and the workspace slots of its partials, in
// key order: slot_of(j) for j < n.  False: nothing to merge (the unit is whole).
struct CombineUnit {
    int s, g, c0, n, first_slot, rg;
    bool ranges;
    __device__ __forceinline__ int slot_of(const Params &p, int j) const {
        return j == 0 ? first_slot : ranges ? 2 * ((c0 + j) * p.rep + rg) : first_slot + j;
    }
};
__device__ __forceinline__ bool combine_unit(const Params &p, CombineUnit &cu) {
    if (p.mode == MODE_UNITS) {
        const int64_t x = p.rb[blockIdx.y + 1], xp = p.rb[blockIdx.y];
        const int64_t u = x >> 32;
        if ((x & 0xffffffffll) == 0 || ((xp >> 32) == u && (xp & 0xffffffffll) != 0)) return false;
        cu.s = (int)(u / p.groups);
        cu.g = (int)(u - (int64_t)cu.s * p.groups);
    } else {
        cu.s = blockIdx.z;
        cu.g = blockIdx.y;
    }
    const StreamPlan &sp = p.st[cu.s];
    int c1;
    cu.rg = cu.g;
    if (p.mode == MODE_RANGES || p.mode == MODE_SPARSE) {
        // the ranges that hold the unit; their CTAs' partial slots
        const int64_t ub = sp.toff, ue = ub + sp.nt;
        cu.c0 = range_of(p, ub);
        c1 = range_of(p, ue - 1);
        cu.first_slot = 2 * (cu.c0 * p.rep + cu.g) + (ub == p.rb[cu.c0] ? 0 : 1);
    } else if (p.mode == MODE_UNITS) {
        // the same over positions (unit, tile), one CTA a range
        const int64_t u = (int64_t)cu.s * p.groups + cu.g;
        const int64_t nt = (unit_keys(sp.len, p.R, p.H, p.ncols, cu.g) + BK - 1) / BK;
        const int64_t ub = unit_pos(u, 0);
        cu.c0 = range_of(p, ub);
        c1 = range_of(p, unit_pos(u, nt - 1));
        cu.rg = 0;
        cu.first_slot = 2 * cu.c0 + (ub == p.rb[cu.c0] ? 0 : 1);
    } else {
        if (p.mode != MODE_SPLITS || sp.nsplit <= 1) return false;
        cu.c0 = 0;
        c1 = sp.nsplit - 1;
        cu.first_slot = sp.slot0 + cu.g * sp.nsplit;
    }
    cu.n = c1 - cu.c0 + 1;
    cu.ranges = p.mode != MODE_SPLITS;
    return cu.n > 1;
}

__device__ __forceinline__ void combine_store(const Params &p, const CombineUnit &cu, int gc, int lane, float M,
                                              float L, const float4 (&acc)[4]) {
    const float inv = 1.f / L;
    const size_t orow = (size_t)cu.s * p.ncols + gc;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(p.out + orow * kLat) + 2 * (lane + 32 * i);
        o2[0] = __floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv);
        o2[1] = __floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv);
    }
    if (lane == 0 && p.lse) p.lse[orow] = (M + log2f(L)) * 0.69314718055994531f;
}

// acc += w * o_j (the column's 512 values, lane's share)
__device__ __forceinline__ void combine_add(float4 (&acc)[4], const float *o, int lane, float w) {
    const float4 *o4 = reinterpret_cast<const float4 *>(o);
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldg(o4 + lane + 32 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[i].x = __fmaf_rn(w, v[i].x, acc[i].x);
        acc[i].y = __fmaf_rn(w, v[i].y, acc[i].y);
        acc[i].z = __fmaf_rn(w, v[i].z, acc[i].z);
        acc[i].w = __fmaf_rn(w, v[i].w, acc[i].w);
    }
}

template <bool WIDE>
__global__ void __launch_bounds__(WIDE ? COMBINE_THREADS : COMBINE_COLS * 32) mla_combine_kernel(const __grid_constant__ Params p) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    CombineUnit cu;
    if (!combine_unit(p, cu)) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = WIDE ? (int)blockIdx.x : (int)blockIdx.x * COMBINE_COLS + warp;   // column of the group
    const int gc = cu.g * NCOL + col;
    if (gc >= p.ncols) return;   // WIDE: the whole block
    const int n = cu.n;
    float4 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if constexpr (!WIDE) {
        // lane j fetches the (m, l) of partial j0 + j; the weights go round by shuffles
        auto ml = [&](int j, float &m, float &l) {
            m = -INFINITY;
            l = 0.f;
            if (j < n) {
                const size_t base = (size_t)cu.slot_of(p, j) * NCOL + col;
                m = __ldg(p.ws_ml + base * 2);
                l = __ldg(p.ws_ml + base * 2 + 1);
            }
        };
        float M = -INFINITY;
        for (int j0 = 0; j0 < n; j0 += 32) {
            float m, l;
            ml(j0 + lane, m, l);
            M = fmaxf(M, m);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        for (int j0 = 0; j0 < n; j0 += 32) {
            float mj, lj;
            ml(j0 + lane, mj, lj);
            const float wj = (mj == -INFINITY) ? 0.f : ptx::ex2(mj - M);
            const int cnt = min(32, n - j0);
#pragma unroll 4
            for (int k = 0; k < cnt; ++k) {
                const float w = __shfl_sync(0xffffffffu, wj, k);
                combine_add(acc, p.ws_o + ((size_t)cu.slot_of(p, j0 + k) * NCOL + col) * kLat, lane, w);
                L = __fmaf_rn(w, __shfl_sync(0xffffffffu, lj, k), L);
            }
        }
        combine_store(p, cu, gc, lane, M, L, acc);
    } else {
        __shared__ float red_m[COMBINE_THREADS / 32];
        __shared__ float red_l[COMBINE_THREADS / 32];
        __shared__ float4 red_o[COMBINE_THREADS / 32][128];
        float m = -INFINITY;
        for (int j = threadIdx.x; j < n; j += COMBINE_THREADS)
            m = fmaxf(m, __ldg(p.ws_ml + ((size_t)cu.slot_of(p, j) * NCOL + col) * 2));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) red_m[warp] = m;
        __syncthreads();
        float M = red_m[0];
#pragma unroll
        for (int w = 1; w < COMBINE_THREADS / 32; ++w) M = fmaxf(M, red_m[w]);
#pragma unroll 2
        for (int j = warp; j < n; j += COMBINE_THREADS / 32) {
            const size_t base = (size_t)cu.slot_of(p, j) * NCOL + col;
            const float mj = __ldg(p.ws_ml + base * 2), lj = __ldg(p.ws_ml + base * 2 + 1);
            const float w = (mj == -INFINITY) ? 0.f : ptx::ex2(mj - M);
            combine_add(acc, p.ws_o + base * kLat, lane, w);
            L = __fmaf_rn(w, lj, L);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) red_o[warp][lane + 32 * i] = acc[i];
        if (lane == 0) red_l[warp] = L;
        __syncthreads();
        if (warp > 0) return;
        float Lt = red_l[0];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = red_o[0][lane + 32 * i];
#pragma unroll
        for (int w = 1; w < COMBINE_THREADS / 32; ++w) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 x = red_o[w][lane + 32 * i];
                acc[i].x += x.x;
                acc[i].y += x.y;
                acc[i].z += x.z;
                acc[i].w += x.w;
            }
            Lt += red_l[w];
        }
        combine_store(p, cu, gc, lane, M, Lt, acc);
    }
}

// ---- host-side plans ----
// RANGES and UNITS: a range holds at least MIN_TILES key tiles, and there are at most as
// many CTAs as the device has SMs.  Launches with more than a quarter as many column
// groups as SMs run UNITS.
struct Plan {
    int mode;
    int64_t total;
    int nranges, rep, nctas;
    size_t slots;   // workspace slots of partials (0: no combine pass)
};

// SPLITS: a function of the stream's own (len, R, H) only.  Splits are whole
// multiples of 256 keys: at most 16 splits of 256..1,024 keys for streams up to 16k
// keys, 1,024-key splits beyond that, and at most 128 splits a stream (a longer
// split) so the partials stay a few percent of the key bytes.  A prefill chunk with
// 128 or more column groups is not split at all.
struct Split {
    int64_t split;
    int nsplit;
};

inline Split split_of(int64_t len, int groups) {
    Split sp;
    if (groups >= 128) {
        sp.split = len;
        sp.nsplit = 1;
        return sp;
    }
    const int64_t units = (len + SPLIT_UNIT - 1) / SPLIT_UNIT;
    int64_t u = (units + 15) / 16;
    u = u < 1 ? 1 : (u > 4 ? 4 : u);
    const int64_t cap = (units + 127) / 128;
    if (cap > u) u = cap;
    sp.split = u * SPLIT_UNIT;
    sp.nsplit = (int)((len + sp.split - 1) / sp.split);
    return sp;
}

constexpr int64_t SEG_COST = 3;   // a prefill unit's start, in key tiles

// RANGES: what a segment start (a query reload, an extra epilogue, the pipeline's refill) weighs
// in key tiles when the ranges are cut, measured on this GPU by sweeping the weight: listed rows
// ran best at 3 (0.476 of HBM against 0.435 at 9), one column group at 5 (decode batch 0.812
// against 0.799 at 3 and 7), two column groups at 12 (the long window 0.560 against 0.526 at 3,
// its last ranges holding the seven short streams).
inline int64_t range_seg_cost(bool sparse, int groups) { return sparse ? 3 : groups == 1 ? 5 : 12; }

// UNITS: cut the units' tiles (stream-major, each unit as many tiles as its last column
// sees) into at most `sms` ranges, writing their bounds b[0..n] as unit_pos values and
// returning n; *cut tells whether a bound falls inside a unit (which leaves partials).
// Weights: a unit's start (a query load, an epilogue) counts SEG_COST tiles.  A bound inside
// a unit of 32 or more tiles lies on one of its eighths, so the CTAs read at no more than
// eight key positions in step (one DRAM read of a tile serves every CTA at its position).
// The ranges are packed greedily up to a load limit, and the limit is the smallest under
// which `n` ranges cover every unit (a binary search), so the longest range is as short as
// the eighths allow.
inline int plan_unit_ranges(int S, int R, int H, int groups, const int64_t *h_len, int sms, int64_t *b, bool *cut) {
    const int64_t units = (int64_t)S * groups;
    const int ncols = R * H;
    std::vector<int64_t> nt(units), w0(units + 1);   // tiles of each unit; weighted start
    w0[0] = 0;
    for (int64_t u = 0; u < units; ++u) {
        const int s = (int)(u / groups);
        nt[u] = (unit_keys(h_len[s], R, H, ncols, (int)(u - (int64_t)s * groups)) + BK - 1) / BK;
        w0[u + 1] = w0[u] + nt[u] + SEG_COST;
    }
    const int64_t W = w0[units];
    auto weight = [&](int64_t x) {
        const int64_t u = x >> 32, t = x & 0xffffffffll;
        return t == 0 ? w0[u] : w0[u] + SEG_COST + t;
    };
    // the furthest allowed bound at weight <= lim (units + 1 past the end: none beyond x)
    auto furthest = [&](int64_t lim) {
        if (lim >= W) return unit_pos(units, 0);
        const int64_t u = (int64_t)(std::upper_bound(w0.begin(), w0.end(), lim) - w0.begin()) - 1;
        const int64_t r = lim - w0[u] - SEG_COST;
        int64_t t = r < 0 ? 0 : (r > nt[u] ? nt[u] : r);
        if (nt[u] >= 32) t = t * 8 / nt[u] * nt[u] / 8;
        return t >= nt[u] ? unit_pos(u + 1, 0) : unit_pos(u, t);
    };
    // ranges needed under a load limit (cap + 1: more than cap)
    auto count = [&](int64_t limit, int cap, int64_t *out) {
        int64_t x = unit_pos(0, 0);
        const int64_t end = unit_pos(units, 0);
        int n = 0;
        if (out) out[0] = x;
        while (x < end) {
            if (n == cap) return cap + 1;
            const int64_t y = furthest(weight(x) + limit);
            if (y <= x) return cap + 1;
            x = y;
            ++n;
            if (out) out[n] = x;
        }
        return n;
    };
    const int64_t want = (W + MIN_TILES - 1) / MIN_TILES;
    int cap = (int)(want < sms ? want : sms);
    if (cap < 1) cap = 1;
    int64_t lo = (W + cap - 1) / cap, hi = W;
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (count(mid, cap, nullptr) <= cap) hi = mid; else lo = mid + 1;
    }
    const int n = count(lo, cap, b);
    *cut = false;
    for (int i = 1; i < n; ++i) *cut |= (b[i] & 0xffffffffll) != 0;
    return n;
}

inline Plan plan_of(int S, int R, int H, const int64_t *h_len, int sms, bool invariant, int64_t *rb = nullptr,
                    bool sparse = false) {
    Plan pl;
    // R * H itself can pass INT32_MAX; callers refuse S * R * H above 2^30, so groups fits an int
    const int groups = (int)(((int64_t)R * H + NCOL - 1) / NCOL);
    pl.slots = 0;
    pl.rep = 1;
    pl.nranges = 0;
    if (invariant) {
        pl.mode = MODE_SPLITS;
        pl.total = 0;
        for (int s = 0; s < S; ++s) {
            const Split sp = split_of(h_len[s], groups);
            pl.total += (int64_t)groups * sp.nsplit;
            if (sp.nsplit > 1) pl.slots += (size_t)groups * sp.nsplit;
        }
        pl.nctas = (int)pl.total;
        return pl;
    }
    if (groups * 4 > sms) {
        pl.mode = MODE_UNITS;
        pl.total = (int64_t)S * groups;
        int64_t rb_local[MAX_CTAS + 1];
        bool cut = false;
        pl.nranges = plan_unit_ranges(S, R, H, groups, h_len, sms, rb ? rb : rb_local, &cut);
        pl.nctas = pl.nranges;
        pl.slots = cut ? 2 * (size_t)pl.nctas : 0;
        return pl;
    }
    pl.mode = MODE_RANGES;
    pl.rep = groups;
    pl.total = 0;
    for (int s = 0; s < S; ++s) pl.total += (h_len[s] + BK - 1) / BK;
    const int64_t want = (pl.total + MIN_TILES - 1) / MIN_TILES;
    const int cap = sms / groups;
    pl.nranges = (int)(want < cap ? want : cap);
    if (pl.nranges < 1) pl.nranges = 1;
    pl.nctas = pl.nranges * pl.rep;
    // Range boundaries.  A range that starts a second stream pays for a query reload
    // and an extra epilogue, about `seg` tiles: a stream's first tile is weighted
    // 1 + seg and the ranges cut the weighted sequence into equal parts.  A cut
    // that lands inside a stream's extra weight moves to the stream's start.
    int64_t rb_local[MAX_CTAS + 1];
    int64_t *b = rb ? rb : rb_local;
    const int64_t seg = range_seg_cost(sparse, groups);
    const int64_t U = pl.total + seg * (int64_t)(S - 1);
    b[0] = 0;
    b[pl.nranges] = pl.total;
    int s = 0;
    int64_t toff = 0;   // first tile of stream s
    for (int i = 1; i < pl.nranges; ++i) {
        const int64_t tau = (int64_t)i * U / pl.nranges;   // weighted position of the cut
        // advance to the last stream whose weighted start is <= tau
        while (s + 1 < S) {
            const int64_t next = toff + (h_len[s] + BK - 1) / BK;
            if (next + seg * (int64_t)(s + 1) > tau) break;
            toff = next;
            ++s;
        }
        const int64_t u0 = toff + seg * (int64_t)s;   // weighted start of stream s
        int64_t x = toff + (tau > u0 ? tau - u0 : 0);
        const int64_t end = toff + (h_len[s] + BK - 1) / BK;
        if (x > end) x = end;
        if (x <= b[i - 1]) x = b[i - 1] + 1;
        const int64_t room = pl.total - (pl.nranges - i);   // leave a tile for every later range
        if (x > room) x = room;
        b[i] = x;
    }
    // a boundary cuts a stream unless it falls between streams
    bool split = false;
    for (int i = 1; i < pl.nranges && !split; ++i) {
        int64_t off = 0;
        for (int ss = 0; ss < S; ++ss) {
            if (b[i] == off) break;
            off += (h_len[ss] + BK - 1) / BK;
            if (b[i] < off) {
                split = true;
                break;
            }
        }
    }
    pl.slots = split ? 2 * (size_t)pl.nctas : 0;
    return pl;
}

inline size_t slot_bytes() { return (size_t)NCOL * kLat * sizeof(float); }

// The most partials any unit of this launch leaves (the combine's form depends on it).
inline int max_partials(const Params &p, const Plan &pl) {
    int most = 1;
    if (pl.mode == MODE_SPLITS) {
        for (int s = 0; s < p.S; ++s) most = std::max(most, (int)p.st[s].nsplit);
    } else if (pl.mode == MODE_UNITS) {
        // consecutive bounds inside one unit
        int run = 0;
        for (int i = 1; i < pl.nranges; ++i) {
            const int64_t x = p.rb[i], xp = p.rb[i - 1];
            const bool inside = (x & 0xffffffffll) != 0;
            run = inside ? (((xp >> 32) == (x >> 32) && (xp & 0xffffffffll) != 0) ? run + 1 : 1) : 0;
            most = std::max(most, run + 1);
        }
    } else {
        for (int s = 0; s < p.S; ++s) {
            const int64_t *b = p.rb, *e = p.rb + pl.nranges + 1;
            const int c0 = (int)(std::upper_bound(b, e, p.st[s].toff) - b) - 1;
            const int c1 = (int)(std::upper_bound(b, e, p.st[s].toff + p.st[s].nt - 1) - b) - 1;
            most = std::max(most, c1 - c0 + 1);
        }
    }
    return most;
}
// On a default pool the partials are at most two slots a CTA; the no-allocation entry point's
// fixed scratch must hold that many, with the (m, l) pairs after them rounded to 256 bytes.
static_assert(2 * (size_t)MAX_CTAS * NCOL * kLat * sizeof(float) +
                      ((2 * (size_t)MAX_CTAS * NCOL * 2 * sizeof(float) + 255) & ~size_t(255)) <=
                  (size_t)TF_STATIC_WS_BYTES,
              "every default-pool call must fit the static scratch");

}  // namespace attn

// SMs of the current device, or an upper bound when no device answers.
static int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                   cudaSuccess || n <= 0) {
        cudaGetLastError();
        return attn::MAX_CTAS;
    }
    return n < attn::MAX_CTAS ? n : attn::MAX_CTAS;
}

size_t attend_workspace_bytes(bool invariant, int S, int R, int H, const int64_t *h_len, bool sparse) {
    const attn::Plan pl = attn::plan_of(S, R, H, h_len, device_sms(), invariant, nullptr, sparse);
    if (pl.slots == 0) return 0;
    const size_t slots = pl.slots;
    const size_t o = slots * attn::slot_bytes();
    const size_t ml = slots * attn::NCOL * 2 * sizeof(float);
    return o + ((ml + 255) & ~size_t(255));
}

// The plan a call would use, for tf_paged_mla_plan_info (host arithmetic only).
int attend_plan_info(int S, int R, int H, const int64_t *h_len, int sms, bool invariant, tf_attend_plan *info,
                     int64_t *range_bounds, int64_t *split_keys) {
    static_assert(TF_PLAN_MAX_RANGES == attn::MAX_CTAS, "the header's bound is the launch's");
    if (sms <= 0) sms = device_sms();
    if (sms > attn::MAX_CTAS) sms = attn::MAX_CTAS;
    int64_t rb[attn::MAX_CTAS + 1];
    const attn::Plan pl = attn::plan_of(S, R, H, h_len, sms, invariant, rb);
    const int groups = (int)(((int64_t)R * H + attn::NCOL - 1) / attn::NCOL);
    info->mode = pl.mode;
    info->ctas = pl.nctas;
    const bool ranged = pl.mode == attn::MODE_RANGES || pl.mode == attn::MODE_UNITS;
    info->nranges = ranged ? pl.nranges : 0;
    info->groups = groups;
    info->work = pl.total;
    info->slots = (int64_t)pl.slots;
    if (range_bounds && ranged)
        for (int i = 0; i <= pl.nranges; ++i) range_bounds[i] = rb[i];
    if (split_keys && pl.mode == attn::MODE_SPLITS)
        for (int s = 0; s < S; ++s) split_keys[s] = attn::split_of(h_len[s], groups).split;
    return TF_OK;
}

// The driver's tensor-map encoder, looked up once: a function-local static is initialised
// exactly once even when several host threads make their first call together.
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

static bool encode(CUtensorMap *tm, void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                   const cuuint32_t *box, CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = get_encode();
    if (!fn) return false;
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(tm, type, rank, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static int ensure_pool_maps(tf_kvpool *pool) {
    std::lock_guard<std::mutex> g(pool->mu);
    if (pool->tmaps_ready) return TF_OK;
    pool->tm_lat.resize(2);
    pool->tm_rope.resize(2);
    const cuuint64_t P = (cuuint64_t)pool->desc.num_pages, C = (cuuint64_t)pool->desc.num_caches;
    if (is_fp8(pool->desc)) {
        // FP8 pages: the codes as bytes, unswizzled 64 x 64 boxes (expanded in shared memory);
        // the rope block as on BF16 pages, at its FP8-page offset.  No row views (no gathers).
        {
            cuuint64_t dims[4] = {(cuuint64_t)kLat, (cuuint64_t)kPageRows, P, C};
            cuuint64_t strides[3] = {(cuuint64_t)kLat, (cuuint64_t)kF8PageBytes, (cuuint64_t)kF8PageBytes * P};
            cuuint32_t box[4] = {64, (cuuint32_t)attn::BK, 1, 1};
            if (!encode(&pool->tm_lat[0], pool->base, 4, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
                return TF_E_CUDA;
        }
        {
            cuuint64_t dims[4] = {(cuuint64_t)kRope, (cuuint64_t)kPageRows, P, C};
            cuuint64_t strides[3] = {(cuuint64_t)kRope * 2, (cuuint64_t)kF8PageBytes, (cuuint64_t)kF8PageBytes * P};
            cuuint32_t box[4] = {64, (cuuint32_t)attn::BK, 1, 1};
            if (!encode(&pool->tm_rope[0], pool->base + kF8RopeOff, 4, dims, strides, box)) return TF_E_CUDA;
        }
        // row views for gathers: 512-byte code rows (644 a page: the scales and the rope block
        // follow, never addressed) and 128-byte rope rows (2,576 a page); one-row boxes
        const cuuint64_t pages = P * C;
        {
            cuuint64_t dims[2] = {(cuuint64_t)kLat, (pages - 1) * (kF8PageBytes / kLat) + kPageRows};
            cuuint64_t strides[1] = {(cuuint64_t)kLat};
            cuuint32_t box[2] = {(cuuint32_t)attn::F8_BLK, 1};
            if (!encode(&pool->tm_lat[1], pool->base, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
                return TF_E_CUDA;
        }
        {
            cuuint64_t dims[2] = {(cuuint64_t)kRope, (pages - 1) * (kF8PageBytes / (kRope * 2)) + kPageRows};
            cuuint64_t strides[1] = {(cuuint64_t)kRope * 2};
            cuuint32_t box[2] = {64, 1};
            if (!encode(&pool->tm_rope[1], pool->base + kF8RopeOff, 2, dims, strides, box)) return TF_E_CUDA;
        }
        pool->tmaps_ready = true;
        return TF_OK;
    }
    {
        cuuint64_t dims[4] = {(cuuint64_t)kLat, (cuuint64_t)kPageRows, P, C};
        cuuint64_t strides[3] = {(cuuint64_t)kLat * 2, (cuuint64_t)kPageBytes, (cuuint64_t)kPageBytes * P};
        cuuint32_t box[4] = {64, (cuuint32_t)attn::BK, 1, 1};
        if (!encode(&pool->tm_lat[0], pool->base, 4, dims, strides, box)) return TF_E_CUDA;
    }
    {
        cuuint64_t dims[4] = {(cuuint64_t)kRope, (cuuint64_t)kPageRows, P, C};
        cuuint64_t strides[3] = {(cuuint64_t)kRope * 2, (cuuint64_t)kPageBytes, (cuuint64_t)kPageBytes * P};
        cuuint32_t box[4] = {64, (cuuint32_t)attn::BK, 1, 1};
        if (!encode(&pool->tm_rope[0], pool->base + kLatBlockBytes, 4, dims, strides, box)) return TF_E_CUDA;
    }
    // row views for gathers: latent rows 1,024 B apart (576 a page, the last 64 of them the
    // rope block, never addressed), rope rows 128 B apart (4,608 a page); one-row boxes
    const cuuint64_t pages = P * C;
    {
        cuuint64_t dims[2] = {(cuuint64_t)kLat, (pages - 1) * (kPageBytes / (kLat * 2)) + kPageRows};
        cuuint64_t strides[1] = {(cuuint64_t)kLat * 2};
        cuuint32_t box[2] = {64, 1};
        if (!encode(&pool->tm_lat[1], pool->base, 2, dims, strides, box)) return TF_E_CUDA;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)kRope, (pages - 1) * (kPageBytes / (kRope * 2)) + kPageRows};
        cuuint64_t strides[1] = {(cuuint64_t)kRope * 2};
        cuuint32_t box[2] = {64, 1};
        if (!encode(&pool->tm_rope[1], pool->base + kLatBlockBytes, 2, dims, strides, box)) return TF_E_CUDA;
    }
    pool->tmaps_ready = true;
    return TF_OK;
}

int launch_attend(tf_kvpool *pool, int cache, const int32_t *d_pt, int max_pages, const int64_t *h_len, int S, int R,
                  int H, const void *d_q, float scale, void *d_out, float *d_lse, void *d_ws, size_t ws_bytes,
                  cudaStream_t st, const int32_t *d_idx, int max_idx, const int32_t *h_nidx) {
    using namespace attn;
    if (prepare_launch(pool, st) != TF_OK) return TF_E_CUDA;
    // every instance opted in to its shared memory once, whichever host thread comes first
    static std::once_flag attr_once;
    static bool attr_ok = false;
    std::call_once(attr_once, [] {
        attr_ok = !(cudaFuncSetAttribute(mla_attend_kernel<MODE_RANGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_TOTAL) != cudaSuccess ||
            cudaFuncSetAttribute(mla_attend_kernel<MODE_UNITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_TOTAL) != cudaSuccess ||
            cudaFuncSetAttribute(mla_attend_kernel<MODE_SPLITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_TOTAL) != cudaSuccess ||
            cudaFuncSetAttribute(mla_attend_kernel<MODE_SPARSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_TOTAL) != cudaSuccess ||
            cudaFuncSetAttribute(mla_attend_kernel<MODE_RANGES, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_TOTAL) != cudaSuccess ||
            cudaFuncSetAttribute(mla_attend_kernel<MODE_UNITS, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_TOTAL) != cudaSuccess ||
            cudaFuncSetAttribute(mla_attend_kernel<MODE_SPARSE, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_TOTAL) != cudaSuccess);
    });
    if (!attr_ok) return TF_E_CUDA;
    int rc = ensure_pool_maps(pool);
    if (rc != TF_OK) return rc;

    // Params is large (tensor maps + the per-stream plan); keep one per host thread.
    thread_local std::unique_ptr<Params> pp;
    if (!pp) pp.reset(new Params());
    Params &p = *pp;
    p.tm_lat = pool->tm_lat[0];
    p.tm_rope = pool->tm_rope[0];
    p.tm_lat_rows = pool->tm_lat[1];
    p.tm_rope_rows = pool->tm_rope[1];
    p.idx = d_idx;
    p.max_idx = max_idx;
    {
        cuuint64_t dims[2] = {(cuuint64_t)kDk, (cuuint64_t)S * R * H};
        cuuint64_t strides[1] = {(cuuint64_t)kDk * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)NCOL};
        if (!encode(&p.tm_q, const_cast<void *>(d_q), 2, dims, strides, box)) return TF_E_CUDA;
    }
    p.pt = d_pt;
    p.q = static_cast<const __nv_bfloat16 *>(d_q);
    p.out = static_cast<__nv_bfloat16 *>(d_out);
    p.lse = d_lse;
    p.err = pool->err;
    p.pool_base = pool->base;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.cache = cache;
    p.max_pages = max_pages;
    p.num_pages = pool->desc.num_pages;
    p.S = S;
    p.R = R;
    p.H = H;
    p.ncols = R * H;
    p.groups = (R * H + NCOL - 1) / NCOL;
    p.windowed = d_pt ? 0 : 1;
    const bool sparse = d_idx != nullptr;
    // the keys of a sparse call are the listed rows: plan over the list lengths
    int64_t nkeys[TF_MAX_STREAMS];
    const int64_t *keys = h_len;
    if (sparse) {
        for (int s = 0; s < S; ++s) nkeys[s] = h_nidx[s];
        keys = nkeys;
    }
    const bool invariant = !sparse && (pool->desc.flags & TF_POOL_BATCH_INVARIANT) != 0;
    Plan pl = plan_of(S, R, H, keys, device_sms(), invariant, p.rb, sparse);
    if (sparse) pl.mode = MODE_SPARSE;   // ranges over the lists (few column groups: R = 1, H <= 128)
    p.mode = pl.mode;
    p.total = pl.total;
    p.nranges = pl.nranges;
    p.rep = pl.rep;
    int64_t off = 0;
    for (int s = 0; s < S; ++s) {
        StreamPlan &sp = p.st[s];
        sp.len = keys[s];
        sp.toff = off;
        sp.nt = (int32_t)((keys[s] + BK - 1) / BK);
        off += sp.nt;
        const Split spl = split_of(keys[s], p.groups);
        sp.split = sparse ? (int32_t)h_len[s] : (int32_t)spl.split;
        sp.nsplit = spl.nsplit;
        sp.item0 = sp.slot0 = sp.pad = 0;
    }
    if (pl.mode == MODE_SPLITS) {
        // launch order: streams with longer splits first, so short work fills the tail;
        // workspace slots follow the caller's order, so their layout does not depend on it
        int order[TF_MAX_STREAMS];
        for (int s = 0; s < S; ++s) order[s] = s;
        std::stable_sort(order, order + S, [&](int a, int b) { return p.st[a].split > p.st[b].split; });
        int items = 0, slots = 0;
        for (int e = 0; e < S; ++e) {
            p.order[e] = (int16_t)order[e];
            p.st[order[e]].item0 = items;
            items += p.groups * p.st[order[e]].nsplit;
        }
        for (int s = 0; s < S; ++s) {
            p.st[s].slot0 = slots;
            if (p.st[s].nsplit > 1) slots += p.groups * p.st[s].nsplit;
        }
    }
    const size_t slots = pl.slots;
    p.ws_o = slots ? static_cast<float *>(d_ws) : nullptr;
    p.ws_ml = slots ? reinterpret_cast<float *>(static_cast<char *>(d_ws) + slots * slot_bytes()) : nullptr;
    (void)ws_bytes;
    {
        ProfScope prof(pool, kProfAttend, st);
        const bool f8 = is_fp8(pool->desc);
        if (f8 && pl.mode == MODE_SPLITS) return TF_E_UNSUPPORTED;
        auto *kern = f8 ? (pl.mode == MODE_RANGES  ? mla_attend_kernel<MODE_RANGES, true>
                           : pl.mode == MODE_UNITS ? mla_attend_kernel<MODE_UNITS, true>
                                                   : mla_attend_kernel<MODE_SPARSE, true>)
                   : pl.mode == MODE_RANGES ? mla_attend_kernel<MODE_RANGES>
                   : pl.mode == MODE_UNITS  ? mla_attend_kernel<MODE_UNITS>
                   : pl.mode == MODE_SPARSE ? mla_attend_kernel<MODE_SPARSE>
                                            : mla_attend_kernel<MODE_SPLITS>;
        const int threads = f8 || pl.mode == MODE_SPARSE ? THREADS + 128 : THREADS;
        const cudaError_t e = launch_pdl(kern, dim3(pl.nctas), dim3(threads), SMEM_TOTAL, st, p);
        launch_counter()++;
        if (e != cudaSuccess) return TF_E_CUDA;
    }
    if (slots) {
        ProfScope prof(pool, kProfCombine, st);
        // UNITS: only the units a range bound cuts
        // UNITS: blockIdx.y runs over the range bounds (only cut units merge)
        const bool wide = max_partials(p, pl) > COMBINE_NARROW_MAX;
        const int groups = (R * H + NCOL - 1) / NCOL;
        const int gx = wide ? NCOL : NCOL / COMBINE_COLS;
        const dim3 grid = pl.mode == MODE_UNITS ? dim3(gx, pl.nranges - 1) : dim3(gx, groups, S);
        const cudaError_t e = launch_pdl(wide ? mla_combine_kernel<true> : mla_combine_kernel<false>, grid,
                                         dim3(wide ? COMBINE_THREADS : COMBINE_COLS * 32), 0, st, p);
        launch_counter()++;
        if (e != cudaSuccess) return TF_E_CUDA;
    }
    return TF_OK;
}

}  // namespace tf
