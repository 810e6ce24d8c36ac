// Internal declarations shared by the host pool code and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/tf_paged_mla.h"

namespace tf {

constexpr int kPageRows = TF_PAGE_ROWS;
constexpr int kLat = TF_LATENT_DIM;
constexpr int kRope = TF_ROPE_DIM;
constexpr int kDk = TF_QK_DIM;
constexpr size_t kLatBlockBytes = size_t(kPageRows) * kLat * 2;   // 524,288
constexpr size_t kRopeBlockBytes = size_t(kPageRows) * kRope * 2; // 65,536
constexpr size_t kPageBytes = kLatBlockBytes + kRopeBlockBytes;   // 589,824
constexpr size_t kCtrlBytes = 256;
// FP8 pages: E4M3 codes, then one fp32 scale a row, then the bf16 rope block.
constexpr size_t kF8LatBlockBytes = size_t(kPageRows) * kLat;         // 262,144
constexpr size_t kF8ScaleOff = kF8LatBlockBytes;
constexpr size_t kF8RopeOff = kF8ScaleOff + size_t(kPageRows) * 4;     // 264,192
constexpr size_t kF8PageBytes = kF8RopeOff + kRopeBlockBytes;          // 329,728
static_assert(kF8PageBytes % 1024 == 0, "FP8 pages keep 1 KiB alignment");

inline bool is_fp8(const tf_kvpool_desc &d) { return (d.flags & TF_POOL_FP8) != 0; }
inline size_t page_bytes(const tf_kvpool_desc &d) { return is_fp8(d) ? kF8PageBytes : kPageBytes; }

// Device error word, in the pool's control block after the last page.
struct DevErr {
    int32_t code;   // 0, TF_E_DEVICE or TF_E_TIMEOUT (first error wins)
    int32_t pad;
    int64_t detail; // offending page id or wait site
};

enum ProfKind { kProfAppend = 0, kProfAttend = 1, kProfCombine = 2, kProfCopy = 3, kProfPoison = 4, kProfKinds = 5 };

struct ProfRec {
    int kind;
    cudaEvent_t a, b;
};

}  // namespace tf

struct tf_kvpool {
    tf_kvpool_desc desc;
    char *base = nullptr;
    size_t bytes = 0;
    tf::DevErr *err = nullptr;  // device address
    std::atomic<bool> err_cleared{false};   // the error word is zeroed before the first launch
    std::vector<int32_t> refcnt;
    std::vector<int32_t> free_ring;  // FIFO of free ids
    size_t free_head = 0, free_count = 0;
    std::mutex mu;
    // TMA descriptors over the pool, one pair (latent, rope) per cache, encoded on first use.
    bool tmaps_ready = false;
    std::vector<CUtensorMap> tm_lat, tm_rope;
    // profiling
    bool prof = false;
    std::vector<tf::ProfRec> recs;
    std::vector<cudaEvent_t> spare_events;
    // FP8 pools on batch-invariant plans: a BF16 view over the workspace that attention expands
    // the rows into, set up and launched under shadow_mu (calls from several host threads)
    tf_kvpool *shadow = nullptr;
    std::mutex shadow_mu;
    ~tf_kvpool() { delete shadow; }
};

namespace tf {

std::atomic<int64_t> &launch_counter();

// Called before every launch.  The first launch on a pool zeroes the device error word and
// waits for it, under the pool's lock, so no launch from any host thread or stream can run
// before the word is clear (a launch queued on another stream could otherwise record an error
// that the zeroing then erases).  Because of that wait the first launch on a pool must not be
// made while its stream is being captured.
inline int prepare_launch(tf_kvpool *pool, cudaStream_t st) {
    if (pool->err_cleared.load(std::memory_order_acquire)) return TF_OK;
    std::lock_guard<std::mutex> g(pool->mu);
    if (pool->err_cleared.load(std::memory_order_relaxed)) return TF_OK;
    if (cudaMemsetAsync(pool->err, 0, sizeof(DevErr), st) != cudaSuccess) return TF_E_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return TF_E_CUDA;
    pool->err_cleared.store(true, std::memory_order_release);
    return TF_OK;
}

// Bracket a launch with profiling events when the pool asks for them.
struct ProfScope {
    tf_kvpool *pool;
    int kind;
    cudaStream_t stream;
    cudaEvent_t a = nullptr, b = nullptr;
    ProfScope(tf_kvpool *p, int k, cudaStream_t s);
    ~ProfScope();
};

// Launch with programmatic stream serialization (see griddep_wait in ptx.cuh).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Kernel launchers (defined in the .cu files).  Arguments are already validated.
int launch_append(tf_kvpool *pool, int cache, const int32_t *d_pt, int max_pages, const int64_t *h_pos,
                  int S, int n, const void *d_lat, const void *d_rope, cudaStream_t st);
int launch_state_copy(tf_kvpool *pool, int cache, const int32_t *d_src, const int32_t *d_dst, int64_t at,
                      cudaStream_t st);
int launch_poison(tf_kvpool *pool, const int32_t *h_ids, int n, cudaStream_t st);
// FP8 pages (fp8.cu).
int launch_append_fp8(tf_kvpool *pool, int cache, const int32_t *d_pt, int max_pages, const int64_t *h_pos,
                      int S, int n, const void *d_lat, const void *d_rope, cudaStream_t st);
int launch_state_copy_fp8(tf_kvpool *pool, int cache, const int32_t *d_src, const int32_t *d_dst, int64_t at,
                          cudaStream_t st);
size_t fp8_shadow_bytes(int S, const int64_t *h_len);
int launch_attend_fp8(tf_kvpool *pool, int cache, const int32_t *d_pt, int max_pages, const int64_t *h_len, int S,
                      int R, int H, const void *d_q, float scale, void *d_out, float *d_lse, void *d_ws,
                      size_t ws_bytes, size_t attend_ws, cudaStream_t st);
int launch_diag_wait(tf_kvpool *pool, long long limit, cudaStream_t st);
size_t attend_workspace_bytes(bool invariant, int S, int R, int H, const int64_t *h_len, bool sparse = false);
int attend_plan_info(int S, int R, int H, const int64_t *h_len, int sms, bool invariant, tf_attend_plan *info,
                     int64_t *range_bounds, int64_t *split_keys);
// d_idx / max_idx / h_nidx: a sparse call (the keys are the listed rows, R = 1), or null.
int launch_attend(tf_kvpool *pool, int cache, const int32_t *d_pt, int max_pages, const int64_t *h_len, int S,
                  int R, int H, const void *d_q, float scale, void *d_out, float *d_lse, void *d_ws,
                  size_t ws_bytes, cudaStream_t st, const int32_t *d_idx = nullptr, int max_idx = 0,
                  const int32_t *h_nidx = nullptr);

}  // namespace tf
