// Host/device interface of the weight-streaming linear kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "engine_layout.h"

namespace mxfp4 {

struct LinearParams {
    const __nv_bfloat16* x;  // [T][K]
    const uint8_t* ws;       // [N][K/32]
    __nv_bfloat16* y;        // [T][N]
    unsigned* status;        // device status word
    int T, K, N;
    int nblk;                // K / 32
    int nkb;                 // ceil(K / 256): weight boxes per row group
    int xcols;               // staged columns per block (= T)
    int cl;                  // CTAs per cluster splitting K (1 = no cluster)
    int tma3d;               // tensor map is the 3D (128 B, rows, K/256) view
    int n_rg;                // ceil(N / 16): row groups
    SmemLayout layout;
};

// Chooses the cluster size (1, 2, 4 or 8 CTAs splitting K) and the shared
// memory plan (whole K per CTA, or K in parts); false if no plan fits.
// units_per_cta = row groups per CTA of the launch (ceil(n_rg / CTAs)).
bool plan_linear(int T, int K, int max_smem, bool few_units, int units_per_cta, int* cl, SmemLayout* L);
cudaError_t launch_linear(const CUtensorMap& tmap, const LinearParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_quantize(const float* w, int64_t n, int64_t k, uint8_t* wq, uint8_t* ws, cudaStream_t stream,
                            int num_sms);

}  // namespace mxfp4
