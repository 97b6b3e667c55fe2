// Host/device interface of the grouped top-k MoE kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mxfp4 {

struct MoeArgs {
    const __nv_bfloat16* x;  // [T][hidden]
    const float* logits;     // [T][E]
    const uint8_t *w1q, *w1s, *w2q, *w2s;
    __nv_bfloat16* y;        // [T][hidden]
    int32_t* topk_ids;       // optional [T][top_k]
    float* topk_w;           // optional [T][top_k]
    void* workspace;
    unsigned* status;
    int T, E, top_k, hidden, inter;
    int n_shared;            // shared experts E .. E + n_shared - 1 of the weight arrays
};

// Workspace of t tokens with kp (token, slot) pairs each (top_k + n_shared).
size_t moe_workspace_bytes(int64_t t, int64_t e, int kp, int64_t hidden, int64_t inter);
int launch_moe(const uint8_t* w1q, const uint8_t* w2q, const MoeArgs& a, int num_sms, int max_smem,
               cudaStream_t stream);

// Tensor maps of packed weights [rows, k/2] (defined with the C ABI). The
// int written is the engine's copy mode (Params::tma3d, see engine.cuh).
int encode_weights(CUtensorMap* map, const uint8_t* wq, int64_t rows, int64_t k, int steps, int* is3d);
int encode_weights_merged_rows(CUtensorMap* map, const uint8_t* wq, int64_t rows, int64_t k, int steps, int box_rows,
                               int* mode);
int encode_weights_gate_up(CUtensorMap* map, const uint8_t* w1q, int64_t experts, int64_t inter, int64_t k, int steps,
                           int* mode);

}  // namespace mxfp4
