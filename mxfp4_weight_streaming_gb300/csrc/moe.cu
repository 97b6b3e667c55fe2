// Grouped top-k MoE decode layer with MXFP4 experts for sm_103a.
//
// What it computes ("Zyphra Inference Wave 2", sections "Kernel Results" and
// "Quantization": at low concurrency a step reads only its tokens' top-k
// routed experts, and each expert receives a few token rows):
//   ids_t = top_k largest logits (descending, ties to the smaller index),
//   g_t   = softmax over the selected logits,
//   h     = SiLU(W1_gate x_t) * (W1_up x_t)         (per routed pair, fp32)
//   y_t   = bf16( sum_j g_tj * W2_{ids_tj} h_tj )   (selection order)
// With shared experts ("Zyphra Inference Wave 2", section "Quantization": a
// token uses its top-k routed experts plus the layer's shared experts) the
// weight arrays hold n_shared more experts after the E routed ones. Every
// token applies each of them after its routed experts, with g = 1: they are
// n_shared more (token, slot) pairs per token, and from the counting sort on
// nothing distinguishes them from routed pairs.
//
// Four launches on the caller's stream:
//   1. route   : one CTA. Top-k + softmax per token (a warp per token), then
//                a deterministic counting sort of the (token, slot) pairs by
//                expert (ascending pair index within an expert), and the
//                chunk tables: each expert's pairs cut into chunks of at
//                most 8 (gate/up) or 4 (down) columns.
//   2. gate/up : weight-streaming engine, one unit = 16 gate rows + the 16
//                matching up rows of one expert for one chunk of tokens;
//                epilogue h = SiLU(a) * b, stored fp32 by sorted pair.
//   3. down    : engine, one unit = 16 W2 rows of one expert; each fp32 h
//                row is staged as two f16 columns (hi + lo, exact to 22
//                bits) that share one power-of-two factor; epilogue stores
//                o = hi + lo partials fp32 by sorted pair.
//   4. combine : y[t][n] = sum over j in order of g_tj * o[pos(t, j)][n].
// Experts no token selects produce no units, so their weights are not read.
// No floating-point atomics anywhere: results are bit-reproducible.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "engine.cuh"
#include "moe_launch.h"
#include "mxfp4.h"

namespace mxfp4 {

constexpr int kChunkGateUp = 8;  // token columns per gate/up chunk
constexpr int kChunkDown = 4;    // pairs per down chunk (two columns each)
constexpr int kRouteThreads = 1024;

// Device pointers into the caller's workspace.
struct MoeWork {
    int* header;  // [0] chunks for gate/up, [1] chunks for down
    int* ids;     // [P] expert of pair p = t*kp + j (kp = top_k + n_shared)
    float* gw;    // [P] gate weight of pair p
    int* pos;     // [P] sorted position of pair p
    int* sorted;  // [P] pair at sorted position
    int* c1_e;    // gate/up chunks: expert, first sorted position, count
    int* c1_start;
    int* c1_cnt;
    int* c2_e;    // down chunks
    int* c2_start;
    int* c2_cnt;
    float* h;     // [P][inter]  by sorted position
    float* o;     // [P][hidden] by sorted position
};

static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

static MoeWork carve(void* base, int64_t P, int64_t hidden, int64_t inter, size_t* total) {
    uint8_t* b = static_cast<uint8_t*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* p = b ? b + off : nullptr;
        off += align256(bytes);
        return p;
    };
    MoeWork w{};
    w.header = reinterpret_cast<int*>(take(256));
    w.ids = reinterpret_cast<int*>(take(P * 4));
    w.gw = reinterpret_cast<float*>(take(P * 4));
    w.pos = reinterpret_cast<int*>(take(P * 4));
    w.sorted = reinterpret_cast<int*>(take(P * 4));
    w.c1_e = reinterpret_cast<int*>(take(P * 4));
    w.c1_start = reinterpret_cast<int*>(take(P * 4));
    w.c1_cnt = reinterpret_cast<int*>(take(P * 4));
    w.c2_e = reinterpret_cast<int*>(take(P * 4));
    w.c2_start = reinterpret_cast<int*>(take(P * 4));
    w.c2_cnt = reinterpret_cast<int*>(take(P * 4));
    w.h = reinterpret_cast<float*>(take(P * inter * 4));
    w.o = reinterpret_cast<float*>(take(P * hidden * 4));
    if (total) *total = off;
    return w;
}

size_t moe_workspace_bytes(int64_t t, int64_t e, int kp, int64_t hidden, int64_t inter) {
    (void)e;
    size_t total = 0;
    carve(nullptr, t * kp, hidden, inter, &total);
    return total;
}

// ------------------------------------------------------------------ route
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// Exclusive scan of one int per thread over a 1024-thread block.
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = warp_tot[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, d);
            if (lane >= d) s += y;
        }
        warp_tot[lane] = s;  // inclusive warp prefix
    }
    __syncthreads();
    const int before = (warp ? warp_tot[warp - 1] : 0) + x - v;
    if (total) *total = warp_tot[31];
    __syncthreads();
    return before;
}

// Top-k of one token's E logits by one warp: lane l holds experts l, l + 32,
// ... (NV per lane, E <= 32 * NV) in registers. Order: larger logit first,
// ties to the smaller index; NaN never beats a number, and if only NaN
// logits remain the smallest free index is taken.
template <int NV>
__device__ __forceinline__ void warp_topk(const float* row, int E, int top_k, int lane, float (&sel_v)[16],
                                          int (&sel_i)[16]) {
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = (lane + 32 * i < E) ? row[lane + 32 * i] : 0.f;
    uint32_t free_mask = 0;  // bit i: expert lane + 32 i exists and is not taken yet
#pragma unroll
    for (int i = 0; i < NV; ++i)
        if (lane + 32 * i < E) free_mask |= 1u << i;
    for (int j = 0; j < top_k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = lane + 32 * i;
            if ((free_mask >> i) & 1u)
                if (better(v[i], c, bv, bi)) {
                    bv = v[i];
                    bi = c;
                }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, d);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi == 0x7fffffff) {  // only NaN logits left: take the smallest free index
            int mine = free_mask ? lane + 32 * (__ffs(free_mask) - 1) : 0x7fffffff;
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) mine = min(mine, __shfl_xor_sync(0xffffffffu, mine, d));
            bi = mine;
            bv = row[bi];
        }
        if ((bi & 31) == lane) free_mask &= ~(1u << (bi >> 5));
        sel_v[j] = bv;
        sel_i[j] = bi;
    }
}

// Pairs: token t's slot j is pair t * kp + j, kp = top_k + n_shared; slots
// j >= top_k are the shared experts E + (j - top_k) with weight 1.
__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_route_kernel(const float* __restrict__ logits, int T, int E, int top_k, int n_shared, MoeWork w,
                     int32_t* topk_ids, float* topk_w) {
    extern __shared__ int route_smem[];
    const int kp = top_k + n_shared;
    const int P = T * kp;
    const int Et = E + n_shared;  // experts in the weight arrays
    int* s_ids = route_smem;  // [P], then two [Et] tables (see below)
    __shared__ int warp_tot[32];
    __shared__ int totals[3];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // Top-k and softmax: one warp per token.
    for (int t = warp; t < T; t += kRouteThreads / 32) {
        const float* row = logits + (size_t)t * E;
        float sel_v[16];
        int sel_i[16];
        if (E <= 256)
            warp_topk<8>(row, E, top_k, lane, sel_v, sel_i);
        else if (E <= 512)
            warp_topk<16>(row, E, top_k, lane, sel_v, sel_i);
        else
            warp_topk<32>(row, E, top_k, lane, sel_v, sel_i);
        if (lane == 0) {
            const float m = sel_v[0];
            float z = 0.f;
            float ex[16];
            for (int j = 0; j < top_k; ++j) {
                ex[j] = expf(sel_v[j] - m);
                z += ex[j];
            }
            for (int j = 0; j < top_k; ++j) {
                const int p = t * kp + j;
                const float g = ex[j] / z;
                s_ids[p] = sel_i[j];
                w.ids[p] = sel_i[j];
                w.gw[p] = g;
                if (topk_ids) topk_ids[t * top_k + j] = sel_i[j];
                if (topk_w) topk_w[t * top_k + j] = g;
            }
            for (int j = 0; j < n_shared; ++j) {
                const int p = t * kp + top_k + j;
                s_ids[p] = E + j;
                w.ids[p] = E + j;
                w.gw[p] = 1.0f;
            }
        }
        __syncwarp();
    }
    __syncthreads();

    // Counting sort by expert; within an expert, pairs keep ascending order.
    int* s_cnt = s_ids + P;   // [Et]: pairs per expert, then the expert's first position
    int* s_run = s_cnt + Et;  // [Et]: pairs of the expert placed so far
    for (int i = threadIdx.x; i < Et; i += kRouteThreads) {
        s_cnt[i] = 0;
        s_run[i] = 0;
    }
    __syncthreads();
    for (int q = threadIdx.x; q < P; q += kRouteThreads) atomicAdd(&s_cnt[s_ids[q]], 1);  // order-free counts
    __syncthreads();
    const int e = threadIdx.x;  // Et <= kRouteThreads (checked by the host)
    const int cnt = e < Et ? s_cnt[e] : 0;
    const int off = block_exclusive_scan(cnt, warp_tot, nullptr);
    const int n1 = (cnt + kChunkGateUp - 1) / kChunkGateUp;
    const int n2 = (cnt + kChunkDown - 1) / kChunkDown;
    const int c1 = block_exclusive_scan(n1, warp_tot, &totals[0]);
    const int c2 = block_exclusive_scan(n2, warp_tot, &totals[1]);
    if (e < Et) s_cnt[e] = off;
    __syncthreads();
    // Positions: one warp walks the pairs in ascending order, 32 at a time;
    // lanes holding the same expert are ranked by lane.
    if (warp == 0) {
        for (int base = 0; base < P; base += 32) {
            const int q = base + lane;
            const bool ok = q < P;
            const int id = ok ? s_ids[q] : -1 - lane;  // distinct ids for idle lanes
            const unsigned peers = __match_any_sync(0xffffffffu, id);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            if (ok) {
                const int at = s_cnt[id] + s_run[id] + rank;
                w.sorted[at] = q;
                w.pos[q] = at;
            }
            __syncwarp();
            if (ok && rank == 0) s_run[id] += __popc(peers);
            __syncwarp();
        }
    }
    if (e < Et && cnt > 0) {
        for (int q = 0; q < n1; ++q) {
            w.c1_e[c1 + q] = e;
            w.c1_start[c1 + q] = off + q * kChunkGateUp;
            w.c1_cnt[c1 + q] = min(kChunkGateUp, cnt - q * kChunkGateUp);
        }
        for (int q = 0; q < n2; ++q) {
            w.c2_e[c2 + q] = e;
            w.c2_start[c2 + q] = off + q * kChunkDown;
            w.c2_cnt[c2 + q] = min(kChunkDown, cnt - q * kChunkDown);
        }
    }
    if (threadIdx.x == 0) {
        w.header[0] = totals[0];
        w.header[1] = totals[1];
    }
}

// --------------------------------------------------------- gate/up (GEMM1)
struct GateUpParams {
    const __nv_bfloat16* x;  // [T][hidden]
    const uint8_t* w1s;      // [E*2*inter][hidden/32]
    MoeWork w;
    unsigned* status;
    int kp, hidden, inter;  // kp: pairs per token (top_k + n_shared)
    int nblk, nkb, xcols, cl, tma3d;
    int upc;                 // units per chunk = inter / 16
    SmemLayout layout;
};

struct GateUpProblem {
    static constexpr int NT = 1;
    static constexpr int BOXES = 2;
    static constexpr int NCW = 11;  // 12 warps: up to 160 registers a thread
    using Params = GateUpParams;

    __device__ static int num_units(const Params& p) { return *(volatile const int*)&p.w.header[0] * p.upc; }
    __device__ static int chunk_of(const Params& p, int u) { return u / p.upc; }
    __device__ static int box_row(const Params& p, int u, int box) {
        const int q = u / p.upc;
        const int j = u - q * p.upc;
        return p.w.c1_e[q] * 2 * p.inter + box * p.inter + 16 * j;
    }
    __device__ static const uint8_t* scale_src(const Params& p, int u, int box) {
        return p.w1s + (size_t)box_row(p, u, box) * p.nblk;
    }
    __device__ static int unit_rows(const Params&, int) { return 16; }
    __device__ static int ncols(const Params& p, int q) { return p.w.c1_cnt[q]; }

    // Staged columns are the chunk's token rows of x (bf16), copied in bulk.
    static constexpr bool kBulkStage = true;
    __device__ static int stage_cols(const Params& p, int q) { return p.w.c1_cnt[q]; }
    __device__ static const uint8_t* stage_row(const Params& p, int q, int col) {
        const int token = p.w.sorted[p.w.c1_start[q] + col] / p.kp;
        return reinterpret_cast<const uint8_t*>(p.x + static_cast<size_t>(token) * p.hidden);
    }

    __device__ static void epilogue(const Params& p, int u, const Sums<1>& v, int lane) {
        const int q = u / p.upc;
        const int j = u - q * p.upc;
        const int cnt = p.w.c1_cnt[q];
        const int start = p.w.c1_start[q];
        for (int e = lane; e < cnt * 16; e += 32) {
            const int t = e >> 4;
            const int r = e & 15;
            const float a = v.sum(0, t, r);
            const float b = v.sum(1, t, r);
            const float silu = a / (1.0f + expf(-a));
            p.w.h[(size_t)(start + t) * p.inter + 16 * j + r] = silu * b;
        }
    }
};

// ------------------------------------------------------------ down (GEMM2)
struct DownParams {
    const uint8_t* w2s;  // [E*hidden][inter/32]
    MoeWork w;
    unsigned* status;
    int hidden, inter;
    int nblk, nkb, xcols, cl, tma3d;
    int upc;             // units per chunk = hidden / 32
    SmemLayout layout;
};

// A unit is 32 W2 rows of one expert (two boxes of 16 rows that share the
// staged h columns): the per-unit costs (scale copy, hand-in, epilogue) are
// spread over twice the weight bytes of a 16-row unit.
struct DownProblem {
    static constexpr int NT = 1;
    static constexpr int BOXES = 2;
    static constexpr int NCW = 11;  // 12 warps: up to 160 registers a thread
    using Params = DownParams;

    __device__ static int num_units(const Params& p) { return *(volatile const int*)&p.w.header[1] * p.upc; }
    __device__ static int chunk_of(const Params& p, int u) { return u / p.upc; }
    __device__ static int box_row(const Params& p, int u, int box) {
        const int q = u / p.upc;
        const int j = u - q * p.upc;
        return p.w.c2_e[q] * p.hidden + 32 * j + 16 * box;
    }
    __device__ static const uint8_t* scale_src(const Params& p, int u, int box) {
        return p.w2s + (size_t)box_row(p, u, box) * p.nblk;
    }
    __device__ static int unit_rows(const Params&, int) { return 16; }
    __device__ static int ncols(const Params& p, int q) { return 2 * p.w.c2_cnt[q]; }

    // Column t holds hi(h_t), column cnt + t holds lo(h_t); staged by the
    // consumer threads from the fp32 rows of h.
    static constexpr bool kBulkStage = false;
    __device__ static void stage(const Params& p, int q, int kblk0, int kblk1, const StageDst& dst, int tid,
                                 int nthreads) {
        const int cnt = p.w.c2_cnt[q];
        const int start = p.w.c2_start[q];
        const int nb = kblk1 - kblk0;
        const int items = nb * cnt;
        for (int it = tid; it < items; it += nthreads) {
            const int b = it / cnt;
            const int t = it - b * cnt;
            const float4* src =
                reinterpret_cast<const float4*>(p.w.h + (size_t)(start + t) * p.inter + (size_t)(kblk0 + b) * 32);
            float v[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 f = src[k];
                v[4 * k] = f.x;
                v[4 * k + 1] = f.y;
                v[4 * k + 2] = f.z;
                v[4 * k + 3] = f.w;
            }
            stage_f32_block_split(v, dst.col(t, b), dst.col(cnt + t, b), dst.factor(t, b), dst.factor(cnt + t, b),
                                  dst.wide);
        }
        for (int it = tid; it < nb * (8 - 2 * cnt); it += nthreads) {
            const int b = it / (8 - 2 * cnt);
            *dst.factor(2 * cnt + (it - b * (8 - 2 * cnt)), b) = 0.0f;
        }
    }

    __device__ static void epilogue(const Params& p, int u, const Sums<1>& v, int lane) {
        const int q = u / p.upc;
        const int j = u - q * p.upc;
        const int cnt = p.w.c2_cnt[q];
        const int start = p.w.c2_start[q];
#pragma unroll
        for (int bx = 0; bx < 2; ++bx)
            for (int e = lane; e < cnt * 16; e += 32) {
                const int t = e >> 4;
                const int r = e & 15;
                p.w.o[(size_t)(start + t) * p.hidden + 32 * j + 16 * bx + r] = v.sum(bx, t, r) + v.sum(bx, cnt + t, r);
            }
    }
};

// ---------------------------------------------------------------- combine
__global__ void moe_combine_kernel(MoeWork w, int T, int kp, int hidden, __nv_bfloat16* __restrict__ y) {
    const int64_t total = (int64_t)T * hidden;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int t = static_cast<int>(i / hidden);
        const int n = static_cast<int>(i - (int64_t)t * hidden);
        float s = 0.f;
        for (int j = 0; j < kp; ++j) {
            const int p = t * kp + j;
            s = fmaf(w.gw[p], w.o[(size_t)w.pos[p] * hidden + n], s);
        }
        y[i] = __float2bfloat16_rn(s);
    }
}

// ------------------------------------------------------------------- host
int launch_moe(const uint8_t* w1q, const uint8_t* w2q, const MoeArgs& a, int num_sms, int max_smem,
               cudaStream_t stream) {
    const int kp = a.top_k + a.n_shared;
    const int64_t P = (int64_t)a.T * kp;
    const int64_t Et = (int64_t)a.E + a.n_shared;
    MoeWork w = carve(a.workspace, P, a.hidden, a.inter, nullptr);

    GateUpParams g{};
    g.x = a.x;
    g.w1s = a.w1s;
    g.w = w;
    g.status = a.status;
    g.kp = kp;
    g.hidden = a.hidden;
    g.inter = a.inter;
    g.nblk = a.hidden / 32;
    g.nkb = (a.hidden + 255) / 256;
    g.xcols = kChunkGateUp;
    g.upc = a.inter / 16;
    g.cl = 1;
    // Gate/up: consumer chunks of half a stage (measured faster than whole
    // stages here: more chunks in flight for the 11 consumer warps).
    const int steps1 = stage_steps(2, g.nkb, 0);
    const int group1 = steps1 % 2 == 0 ? steps1 / 2 : steps1;
    if (!plan_layout(1, 2, g.nblk, g.nblk, g.xcols, 1, GateUpProblem::NCW, kRedStride, steps1, group1, g.nkb,
                     max_smem, &g.layout))
        return MXFP4_ERR_SHAPE;

    DownParams d{};
    d.w2s = a.w2s;
    d.w = w;
    d.status = a.status;
    d.hidden = a.hidden;
    d.inter = a.inter;
    d.nblk = a.inter / 32;
    d.nkb = (a.inter + 255) / 256;
    d.xcols = 2 * kChunkDown;
    d.upc = a.hidden / 32;
    d.cl = 1;
    // Down: a consumer warp takes whole stages (measured faster than half
    // stages here; gate/up is faster with half stages).
    const int steps2 = stage_steps(2, d.nkb, 0);
    const int group2 = steps2;
    if (!plan_layout(1, 2, d.nblk, d.nblk, d.xcols, 1, DownProblem::NCW, kRedStride, steps2, group2, d.nkb,
                     max_smem, &d.layout))
        return MXFP4_ERR_SHAPE;

    CUtensorMap map1, map2;
    // One copy per stage: an expert's 16 gate rows with their 16 up rows, and
    // 32 consecutive W2 rows.
    if (int rc = encode_weights_gate_up(&map1, w1q, Et, a.inter, a.hidden, static_cast<int>(g.layout.steps), &g.tma3d))
        return rc;
    if (int rc = encode_weights_merged_rows(&map2, w2q, Et * a.hidden, a.inter, static_cast<int>(d.layout.steps), 32,
                                            &d.tma3d))
        return rc;

    const int route_smem = static_cast<int>((P + 2 * Et) * 4);
    if (route_smem > 48 * 1024) {
        if (cudaFuncSetAttribute(moe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, route_smem) !=
            cudaSuccess)
            return MXFP4_ERR_CUDA;
    }
    moe_route_kernel<<<1, kRouteThreads, route_smem, stream>>>(a.logits, a.T, a.E, a.top_k, a.n_shared, w,
                                                               a.topk_ids, a.topk_w);
    if (cudaGetLastError() != cudaSuccess) return MXFP4_ERR_CUDA;
    // The unit counts are only known on the device; launch one CTA per SM.
    if (launch_stream_kernel<GateUpProblem>(map1, g, num_sms, num_sms, stream) != cudaSuccess) return MXFP4_ERR_CUDA;
    if (launch_stream_kernel<DownProblem>(map2, d, num_sms, num_sms, stream) != cudaSuccess) return MXFP4_ERR_CUDA;
    const int64_t total = (int64_t)a.T * a.hidden;
    int blocks = static_cast<int>((total + 255) / 256);
    if (blocks > num_sms * 8) blocks = num_sms * 8;
    moe_combine_kernel<<<blocks, 256, 0, stream>>>(w, a.T, kp, a.hidden, a.y);
    return cudaGetLastError() == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}

}  // namespace mxfp4
