// Host interface of the packed-E2M1 tensor-core linear kernel (f4_linear.cu):
// tcgen05.mma kind::mxf4 with the weights as stored and the activations as
// eight E2M1 digit pieces, for 1 <= t <= 16.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mxfp4 {
namespace f4 {

struct F4Params {
    const __nv_bfloat16* x;  // [T, K] (unused when xab is set)
    const float* xab;        // when set: activations SiLU(xab[t, k]) * xab[t, K + k], rows of 2K floats
    const uint8_t* ws;       // [N, K/32] E8M0
    __nv_bfloat16* y;        // [T, N] (unused when yf is set)
    float* yf;               // when set: fp32 outputs [T, N] instead of y
    unsigned* status;        // device status word (bounded-wait timeouts)
    int T, K, N;
    int nblk;       // K / 32
    int stages;     // K / 512: stages over all of K
    int rows;       // rows per group (a multiple of 8); group g owns [g*rows, (g+1)*rows)
    int h_main;     // rows of every tile but a group's last (min(rows, 128))
    int h_tail;     // rows of a group's last tile when rows % 128 != 0 and rows > 128, else 0
    int cl;         // CTAs per cluster splitting K (1 or 2)
    int na;         // weight ring slots
    int nb;         // activation (digit piece) buffers
    int max_batch;  // tiles whose accumulators fit in TMEM at once
    int tmem_cols;  // TMEM columns the CTA allocates (256 or 512)
    int inbox_bytes;  // rank 0's inbox for rank 1's sums (cluster of 2: tiles x 128 rows x 16-byte vectors), else 0
};

// How a call is cut (host only).
struct F4Plan {
    int npad;        // MMA N: 8 pieces x t, rounded up to 16, 32, 48 or 64
    int cl;          // cluster size
    int grid;        // CTAs launched
    int groups;      // row groups (clusters or lone CTAs)
    int rows;        // rows per group
    int h_main, h_tail;
    int tiles;       // tiles per group (at most)
    int na;          // weight ring slots
    int nb;          // activation buffers
    int max_batch;
    int tmem_cols;
    int inbox_bytes;
    int smem_bytes;  // dynamic shared memory per CTA, as launched
};

// False when the shape is outside the kernel's limits (t > 16, k % 512 != 0,
// no shared-memory fit, or t > 8 with a CTA's tiles not in one batch). swiglu_in: the plan of a call with xab set, for
// t <= 4 only (its conversion holds four loads per unit, two stages ahead:
// one CTA per SM, and more tokens would spill).
bool plan_f4(int t, int64_t k, int64_t n, int num_sms, int max_smem, F4Plan* out, bool swiglu_in = false);

// main_map / tail_map: the packed codes as the 3D view (128 B, rows, k/256)
// with boxes of (128 B, h_main, 2) and (128 B, h_tail, 2) (tail_map unused
// when h_tail == 0).
cudaError_t launch_f4_linear(const CUtensorMap& main_map, const CUtensorMap& tail_map, const F4Params& p,
                             const F4Plan& plan, cudaStream_t stream);

}  // namespace f4
}  // namespace mxfp4
