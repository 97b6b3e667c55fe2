// mxfp4_moe_noalloc: the grouped top-k MoE layer without a caller-supplied
// workspace.
//
// Who needs it: callers that cannot allocate device memory where they run
// the layer. Examples are a plugin inside a framework whose memory pool
// already owns the device memory, so a raw cudaMalloc can fail or fragment
// it; serving loops that forbid allocation after warm-up so their memory
// footprint stays fixed; and latency-bound decode loops that cannot afford
// cudaMalloc's implicit device synchronisation. For them the scratch that
// mxfp4_moe takes from its `workspace` argument lives here instead, in one
// fixed array in device memory.
//
// Costs and rules:
//   * The array is MXFP4_MOE_NOALLOC_SCRATCH_BYTES (12 MiB) on every GPU that
//     loads this library, held until the process exits.
//   * Problems whose scratch exceeds it are rejected with
//     MXFP4_ERR_WORKSPACE before anything is launched.
//   * The first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current); make that first call
//     before any stream capture. Later calls only read the cached address.
//   * All calls share the array and it keeps the last call's contents. The
//     MoE kernels write every scratch byte they read earlier in the same
//     call, so nothing needs clearing; but calls that overlap on the GPU
//     (different streams without ordering between them) race on it.
//   * No cudaMalloc, cudaFree or other allocating routine is called.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mxfp4.h"

namespace {

static __device__ __align__(256) uint8_t g_moe_scratch[MXFP4_MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_moe_scratch on the current device (looked up once per
// device; the host-side symbol itself is not a device address).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MXFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_moe_scratch) != cudaSuccess || !ptr) return MXFP4_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return MXFP4_OK;
}

}  // namespace

extern "C" int mxfp4_moe_noalloc(const void* x, int64_t t, int64_t hidden, const float* router_logits, int64_t e,
                                 int top_k, const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q,
                                 const uint8_t* w2s, int64_t inter, void* y, int32_t* topk_ids, float* topk_w,
                                 void* stream) {
    const size_t need = mxfp4_moe_workspace_size(t, e, top_k, hidden, inter);
    if (need > MXFP4_MOE_NOALLOC_SCRATCH_BYTES) return MXFP4_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (int rc = scratch_address(&scratch)) return rc;
    return mxfp4_moe(x, t, hidden, router_logits, e, top_k, w1q, w1s, w2q, w2s, inter, y, topk_ids, topk_w, scratch,
                     MXFP4_MOE_NOALLOC_SCRATCH_BYTES, stream);
}
