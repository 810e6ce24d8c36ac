// tf_paged_mla_attend_static: the attention call for callers that cannot allocate
// device memory, with the split partials in a file-scope device array instead of a
// caller workspace.  Everything else is tf_paged_mla_attend, called unchanged.
#include <mutex>

#include "tf_internal.h"

namespace {

// The scratch every call of this entry point shares.  Each GPU that loads the
// library holds TF_STATIC_WS_BYTES of it until the process exits.  On the host this
// name is only a stand-in: kernels get the device address from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_static_ws[TF_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_ws_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device
// (with that device current) and remembered.  nullptr if the lookup fails.
void *static_ws_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_ws_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) {
            cudaGetLastError();   // leave no sticky error behind for the caller's next CUDA check
            return nullptr;
        }
        g_ws_addr[dev] = p;
    }
    return g_ws_addr[dev];
}

}  // namespace

extern "C" int tf_paged_mla_attend_static(tf_kvpool *pool, int32_t cache, const int32_t *d_pt, int32_t max_pages,
                                          const int64_t *h_len, int32_t S, int32_t R, int32_t H, const void *d_q,
                                          float scale, void *d_out, float *d_lse, void *cuda_stream) {
    if (!pool || !h_len || S < 1 || S > TF_MAX_STREAMS || R < 1 || H < 1 || H > TF_MAX_HEADS) return TF_E_ARG;
    if ((int64_t)S * R * H > (int64_t)1 << 30) return TF_E_UNSUPPORTED;   // as tf_paged_mla_attend, before sizing
    // FP8 pages on a batch-invariant pool are expanded in a caller workspace
    if (tf::is_fp8(pool->desc) && (pool->desc.flags & TF_POOL_BATCH_INVARIANT)) return TF_E_UNSUPPORTED;
    for (int s = 0; s < S; ++s)
        if (h_len[s] < R) return TF_E_RANGE;
    const size_t need = tf_paged_mla_workspace_bytes(pool, S, R, H, h_len);
    if (need > (size_t)TF_STATIC_WS_BYTES) return TF_E_NOMEM;
    void *ws = nullptr;
    if (need > 0) {
        ws = static_ws_on_current_device();
        if (!ws) return TF_E_CUDA;
    }
    return tf_paged_mla_attend(pool, cache, d_pt, max_pages, h_len, S, R, H, d_q, scale, d_out, d_lse, ws,
                               need > 0 ? (size_t)TF_STATIC_WS_BYTES : 0, cuda_stream);
}
