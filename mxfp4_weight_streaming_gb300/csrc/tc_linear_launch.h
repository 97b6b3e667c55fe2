// Host interface of the block-scaled tensor-core linear kernel (tc_linear.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mxfp4 {
namespace tc {

struct TcLinearParams {
    const __nv_bfloat16* x;  // [T, K]
    const uint8_t* ws;       // [N, K/32] E8M0
    __nv_bfloat16* y;        // [T, N]
    unsigned* status;        // device status word (bounded-wait timeouts)
    int T, K, N;
    int nblk;    // K / 32
    int stages;  // K stages of one row (atoms_per_stage atoms of 128 values)
    int tiles;   // ceil(N / 128)
    int cl;      // CTAs per cluster splitting K (then one tile per cluster)
};

// How a call is cut (host only).
struct TcPlan {
    int cl;               // cluster size (1 or 2)
    int grid;             // CTAs launched
    int atoms_per_stage;  // 128-value atoms per TMA copy / pipeline stage
    int stages;           // stages over all of K
    int tiles;            // 128-row tiles
    int ring_slots;       // weight stages in flight
    int smem_bytes;       // dynamic shared memory per CTA (with alignment slack)
};

// False when the shape is outside the kernel's limits (t > 32, k % 512 !=
// 0, or no shared-memory fit). k % 512 keeps each 4-atom group of a row's
// scale bytes 16-byte aligned (one vector load per row).
bool plan_tc(int t, int64_t k, int64_t n, int num_sms, int max_smem, TcPlan* out);

// atoms_per_stage(t, cl): the stage size plan_tc picks for t tokens and
// cluster size cl (the tensor map's box depth).
int atoms_per_stage(int t, int cl);

// amap: the packed codes (16U4_ALIGN16B, 3D, box 128 values x 128 rows x
// atoms_per_stage).
cudaError_t launch_tc_linear(const CUtensorMap& amap, const TcLinearParams& p, const TcPlan& plan,
                             cudaStream_t stream);

}  // namespace tc
}  // namespace mxfp4
