// Fused dense FFN chain: up -> SwiGLU -> down in one persistent launch.
//
// What it computes (a dense SwiGLU feed-forward block, the MoE expert's
// arithmetic of "Zyphra Inference Wave 2", section "Kernel Results", applied
// to every token with weight 1; fused into one kernel in the direction of
// the megakernels of lithosai "Low-Latency Inference on AMD MI355X" and AMD
// "megakernel-intro", section "1. Megakernels", where SMs that finish early
// preload the weights of the next stage):
//   a = W1[0:inter] x_t (gate rows), b = W1[inter:2*inter] x_t (up rows),
//   h_t = SiLU(a) * b                 (fp32, kept in the workspace)
//   y_t = bf16( W2 h_t )
//
// One CTA per SM, cooperative launch (every CTA is resident, so a CTA may
// wait for the others). Each CTA runs the weight-streaming engine twice on
// the same shared memory:
//   phase A: units of 16 gate + 16 up rows over K = hidden, x staged once;
//            the epilogue stores h and counts the unit in a device word.
//   phase B: units of 16 W2 rows over K = inter. The producer starts
//            streaming W2 as soon as its CTA has finished phase A; the
//            consumers wait (bounded) until every CTA's phase-A units are
//            counted, then stage h as two f16 columns per token (hi + lo,
//            exact to 22 bits, sharing one power-of-two factor).
// The counter is zeroed by the host before each launch (one 4-byte memset on
// the stream). No floating-point atomics: results are bit-reproducible.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "engine.cuh"
#include "ffn_launch.h"
#include "moe_launch.h"
#include "mxfp4.h"

namespace mxfp4 {

namespace {

// ------------------------------------------------------------ phase A
struct FfnUpParams {
    const __nv_bfloat16* x;  // [T][hidden]
    const uint8_t* w1s;      // [2*inter][hidden/32]
    float* h;                // [T][inter]
    unsigned* done;          // phase-A units finished (zeroed before the launch)
    unsigned* status;
    int T, hidden, inter;
    int nblk, nkb, xcols, cl, tma3d;
    SmemLayout layout;
};

struct FfnUpProblem {
    static constexpr int NT = 1;
    static constexpr int BOXES = 2;
    static constexpr int NCW = 11;
    using Params = FfnUpParams;

    __device__ static int num_units(const Params& p) { return p.inter / 16; }
    __device__ static int chunk_of(const Params&, int) { return 0; }
    __device__ static int box_row(const Params& p, int u, int box) { return box * p.inter + 16 * u; }
    __device__ static const uint8_t* scale_src(const Params& p, int u, int box) {
        return p.w1s + (size_t)box_row(p, u, box) * p.nblk;
    }
    __device__ static int unit_rows(const Params&, int) { return 16; }
    __device__ static int ncols(const Params& p, int) { return p.T; }

    static constexpr bool kBulkStage = true;
    __device__ static int stage_cols(const Params& p, int) { return p.T; }
    __device__ static const uint8_t* stage_row(const Params& p, int, int col) {
        return reinterpret_cast<const uint8_t*>(p.x + static_cast<size_t>(col) * p.hidden);
    }

    __device__ static void epilogue(const Params& p, int u, const Sums<1>& v, int lane) {
        for (int e = lane; e < p.T * 16; e += 32) {
            const int t = e >> 4;
            const int r = e & 15;
            const float a = v.sum(0, t, r);
            const float b = v.sum(1, t, r);
            const float silu = a / (1.0f + expf(-a));
            p.h[(size_t)t * p.inter + 16 * u + r] = silu * b;
        }
        // Publish the unit: every lane's stores, then one release count.
        __threadfence();
        __syncwarp();
        if (lane == 0) atom_add_release_gpu(p.done, 1u);
    }
};

// ------------------------------------------------------------ phase B
struct FfnDownParams {
    const uint8_t* w2s;     // [hidden][inter/32]
    const float* h;         // [T][inter], written by phase A of every CTA
    const unsigned* done;   // phase-A units finished
    unsigned* status;
    __nv_bfloat16* y;       // [T][hidden]
    int T, hidden, inter;
    unsigned up_units;      // phase-A units in all (inter / 16)
    int nblk, nkb, xcols, cl, tma3d;
    SmemLayout layout;
};

template <int NT_>
struct FfnDownProblem {
    static constexpr int NT = NT_;
    // 16-row units: hidden / 16 of them spread evenly over the SMs (32-row
    // units left a third of the CTAs with one unit less than the rest), and
    // the smaller stages leave more ring slots beside the staged h.
    static constexpr int BOXES = 1;
    static constexpr int NCW = 11;
    using Params = FfnDownParams;

    __device__ static int num_units(const Params& p) { return p.hidden / 16; }
    __device__ static int chunk_of(const Params&, int) { return 0; }
    __device__ static int box_row(const Params&, int u, int) { return 16 * u; }
    __device__ static const uint8_t* scale_src(const Params& p, int u, int box) {
        return p.w2s + (size_t)box_row(p, u, box) * p.nblk;
    }
    __device__ static int unit_rows(const Params&, int) { return 16; }
    __device__ static int ncols(const Params& p, int) { return 2 * p.T; }

    // h comes from phase A of every CTA: wait until all of it is counted.
    static constexpr bool kInputGate = true;
    __device__ static bool wait_inputs(const Params& p, const WaitCtx& wc) {
        int ok = 1;
        if ((threadIdx.x & 31) == 0) ok = wait_global_at_least(p.done, p.up_units, wc);  // one poller a warp
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __threadfence();  // every lane's later loads of h come after the count it saw
        return ok != 0;
    }

    // Column t holds hi(h_t), column T + t holds lo(h_t).
    static constexpr bool kBulkStage = false;
    __device__ static void stage(const Params& p, int, int kblk0, int kblk1, const StageDst& dst, int tid,
                                 int nthreads) {
        const int T = p.T;
        const int nb = kblk1 - kblk0;
        for (int it = tid; it < nb * T; it += nthreads) {
            const int b = it / T;
            const int t = it - b * T;
            // L2 loads: h was written by other SMs during this launch.
            const float4* src = reinterpret_cast<const float4*>(p.h + (size_t)t * p.inter + (size_t)(kblk0 + b) * 32);
            float v[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 f = __ldcg(src + k);
                v[4 * k] = f.x;
                v[4 * k + 1] = f.y;
                v[4 * k + 2] = f.z;
                v[4 * k + 3] = f.w;
            }
            stage_f32_block_split(v, dst.col(t, b), dst.col(T + t, b), dst.factor(t, b), dst.factor(T + t, b),
                                  dst.wide);
        }
        const int unused = 8 * NT - 2 * T;
        for (int it = tid; it < nb * unused; it += nthreads) {
            const int b = it / unused;
            *dst.factor(2 * T + (it - b * unused), b) = 0.0f;
        }
    }

    __device__ static void epilogue(const Params& p, int u, const Sums<NT>& v, int lane) {
        for (int e = lane; e < p.T * 16; e += 32) {
            const int t = e >> 4;
            const int r = e & 15;
            const float s = v.sum(0, t, r) + v.sum(0, p.T + t, r);
            p.y[(size_t)t * p.hidden + 16 * u + r] = __float2bfloat16_rn(s);
        }
    }
};

static_assert(Roles<FfnUpProblem>::kThreads == Roles<FfnDownProblem<1>>::kThreads &&
                  Roles<FfnUpProblem>::kThreads == Roles<FfnDownProblem<2>>::kThreads,
              "both phases run on the same CTA");

template <int NT2>
__global__ void __launch_bounds__(Roles<FfnUpProblem>::kThreads, 1)
    ffn_chain_kernel(const __grid_constant__ CUtensorMap map1, const __grid_constant__ CUtensorMap map2,
                     const FfnUpParams up, const FfnDownParams down) {
    extern __shared__ uint8_t smem_raw[];
    stream_body<FfnUpProblem, false>(map1, up, smem_raw);
    __syncthreads();
    const bool aborted = stream_smem_release(up.layout, smem_raw, false);
    fence_proxy_async_shared();  // phase A's reads of the ring come before phase B's copies into it
    __syncthreads();
    // A CTA that gave up in phase A stops; the others' phase-B waits for its
    // units then give up too (bounded), and the status word says so.
    if (aborted) return;
    stream_body<FfnDownProblem<NT2>, false>(map2, down, smem_raw);
}

template <int NT2>
cudaError_t launch_chain(const CUtensorMap& map1, const CUtensorMap& map2, const FfnUpParams& up,
                         const FfnDownParams& down, int smem, int grid, cudaStream_t stream) {
    static int configured[64] = {0};  // dynamic smem already allowed, per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || configured[dev] < smem) {
        cudaError_t e = cudaFuncSetAttribute(ffn_chain_kernel<NT2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = smem;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ffn_chain_kernel<NT2>,
                                                                 Roles<FfnUpProblem>::kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Roles<FfnUpProblem>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // Every CTA waits for the phase-A units of all the others: they must all
    // be resident at once.
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, ffn_chain_kernel<NT2>, map1, map2, up, down);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

// A counter word (then h, fp32 [t, inter]) for the cooperative kernel, or
// a | b (fp32 [t, 2 inter]) for the two-launch chain: both from byte 256.
size_t ffn_workspace_bytes(int64_t t, int64_t inter) { return 256 + align256(static_cast<size_t>(t * inter) * 8); }

int plan_ffn(int t, int hidden, int inter, int max_smem, FfnPlan* out) {
    FfnPlan pl{};
    const int nblk1 = hidden / 32, nkb1 = (hidden + 255) / 256;
    const int nblk2 = inter / 32, nkb2 = (inter + 255) / 256;
    // Gate/up: consumer chunks of half a stage; down: whole stages (the
    // grouped MoE's measured choices for the same two problems).
    const int steps1 = stage_steps(2, nkb1, 0);
    const int group1 = steps1 % 2 == 0 ? steps1 / 2 : steps1;
    const int steps2 = stage_steps(1, nkb2, 0);
    pl.nt2 = 2 * t <= 8 ? 1 : 2;
    if (!plan_layout(1, 2, nblk1, nblk1, t, 1, FfnUpProblem::NCW, kRedStride, steps1, group1, nkb1, max_smem,
                     &pl.up))
        return MXFP4_ERR_SHAPE;
    if (!plan_layout(pl.nt2, 1, nblk2, nblk2, 2 * t, 1, FfnUpProblem::NCW, kRedStride, steps2, steps2, nkb2,
                     max_smem, &pl.down))
        return MXFP4_ERR_SHAPE;
    const uint32_t total = pl.up.total > pl.down.total ? pl.up.total : pl.down.total;
    pl.smem_bytes = static_cast<int>(total) + 1024;
    if (pl.smem_bytes > max_smem) return MXFP4_ERR_SHAPE;
    *out = pl;
    return MXFP4_OK;
}

int launch_ffn(const FfnArgs& a, int num_sms, int max_smem, cudaStream_t stream) {
    FfnPlan pl{};
    if (int rc = plan_ffn(a.T, a.hidden, a.inter, max_smem, &pl)) return rc;
    unsigned* done = static_cast<unsigned*>(a.workspace);
    float* h = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + 256);

    FfnUpParams up{};
    up.x = a.x;
    up.w1s = a.w1s;
    up.h = h;
    up.done = done;
    up.status = a.status;
    up.T = a.T;
    up.hidden = a.hidden;
    up.inter = a.inter;
    up.nblk = a.hidden / 32;
    up.nkb = (a.hidden + 255) / 256;
    up.xcols = a.T;
    up.cl = 1;
    up.layout = pl.up;

    FfnDownParams down{};
    down.w2s = a.w2s;
    down.h = h;
    down.done = done;
    down.status = a.status;
    down.y = a.y;
    down.T = a.T;
    down.hidden = a.hidden;
    down.inter = a.inter;
    down.up_units = static_cast<unsigned>(a.inter / 16);
    down.nblk = a.inter / 32;
    down.nkb = (a.inter + 255) / 256;
    down.xcols = 2 * a.T;
    down.cl = 1;
    down.layout = pl.down;

    CUtensorMap map1, map2;
    if (int rc = encode_weights_gate_up(&map1, a.w1q, 1, a.inter, a.hidden, static_cast<int>(pl.up.steps), &up.tma3d))
        return rc;
    if (int rc = encode_weights(&map2, a.w2q, a.hidden, a.inter, static_cast<int>(pl.down.steps), &down.tma3d))
        return rc;

    const int units = a.inter / 16 > a.hidden / 16 ? a.inter / 16 : a.hidden / 16;
    const int grid = units < num_sms ? units : num_sms;
    if (cudaMemsetAsync(done, 0, sizeof(unsigned), stream) != cudaSuccess) return MXFP4_ERR_CUDA;
    const cudaError_t e = pl.nt2 == 1 ? launch_chain<1>(map1, map2, up, down, pl.smem_bytes, grid, stream)
                                      : launch_chain<2>(map1, map2, up, down, pl.smem_bytes, grid, stream);
    return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}

}  // namespace mxfp4
