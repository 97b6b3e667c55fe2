// Host/device interface of the fused dense FFN chain (up -> SwiGLU -> down).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "engine_layout.h"

namespace mxfp4 {

struct FfnArgs {
    const __nv_bfloat16* x;  // [T][hidden]
    const uint8_t *w1q, *w1s, *w2q, *w2s;
    __nv_bfloat16* y;        // [T][hidden]
    void* workspace;         // ffn_workspace_bytes(T, inter), 256-byte aligned
    unsigned* status;
    int T, hidden, inter;
};

// Shared-memory plans of the two phases; the CTA takes the larger.
struct FfnPlan {
    SmemLayout up, down;
    int nt2;         // 8-column token tiles of the down phase (2T columns)
    int smem_bytes;  // dynamic shared memory per CTA, as launched
};

size_t ffn_workspace_bytes(int64_t t, int64_t inter);
int plan_ffn(int t, int hidden, int inter, int max_smem, FfnPlan* out);
int launch_ffn(const FfnArgs& a, int num_sms, int max_smem, cudaStream_t stream);

}  // namespace mxfp4
