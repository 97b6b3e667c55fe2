// C ABI of the MXFP4 weight-streaming library: argument checks, per-device
// set-up (SM count, shared-memory limit, status word), TMA descriptors and
// kernel launches. Every compute step runs in this library's kernels.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "device_common.cuh"
#include "linear_launch.h"
#include "ffn_launch.h"
#include "moe_launch.h"
#include "tc_linear_launch.h"
#include "f4_linear_launch.h"
#include "mxfp4.h"

namespace {

// Per-device status word: kernels OR in mxfp4::kStatusTimeout when a bounded
// wait gives up. Read and cleared by mxfp4_last_device_status().
__device__ unsigned g_status_word;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    int max_smem = 0;
    unsigned* status = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MXFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MXFP4_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return MXFP4_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return MXFP4_ERR_CUDA;
        d.status = static_cast<unsigned*>(p);
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return MXFP4_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    *out = &d;
    return MXFP4_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Packed weights [rows, k/2] as a TMA tensor map with the 128-byte swizzle.
// With k % 256 == 0 the map is the 3D view (128 B, rows, k/256 segments of
// 128 B): one copy lands `steps` segments of 16 rows as [step][row][128 B].
// Otherwise it is the 2D view (k/2 B, rows) fetched one 16 x 128-byte box at
// a time (the 3D view would let the last segment of the last row run past
// the end of the array). Returns whether the 3D view was used in *is3d.
int encode_weight_map(CUtensorMap* map, const uint8_t* wq, int64_t rows, int64_t k, int steps, int* is3d) {
    CUresult r;
    if (k % 256 == 0) {
        cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(k / 256)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(k / 2), 128};
        cuuint32_t box[3] = {128, 16, static_cast<cuuint32_t>(steps)};
        cuuint32_t estride[3] = {1, 1, 1};
        r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(wq), dims, strides, box, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r == CUDA_SUCCESS) {
            *is3d = 1;
            return MXFP4_OK;
        }
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(k / 2), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(k / 2)};
    cuuint32_t box[2] = {128, 16};
    cuuint32_t estride[2] = {1, 1};
    r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(wq), dims, strides, box, estride,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *is3d = 0;
    return r == CUDA_SUCCESS ? MXFP4_OK : MXFP4_ERR_CUDA;
}

// Packed weights [rows, k/2] for the block-scaled tensor-core kernel: the
// 16U4_ALIGN16B type unpacks 16 codes per 16 bytes of shared memory (8 bytes
// of codes, 8 of gap), the layout the MMA reads E2M1 in. The 3D view
// (128 values, rows, k/128 atoms) with strides (k/2 B, 64 B) lets one copy
// fetch `atoms` consecutive atoms of 128 rows: [atom][row][128 B], swizzled.
// Needs wq 32-byte aligned and k % 128 == 0.
int encode_tc_weight_map(CUtensorMap* map, const uint8_t* wq, int64_t rows, int64_t k, int atoms) {
    cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(k / 128)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(k / 2), 64};
    cuuint32_t box[3] = {128, 128, static_cast<cuuint32_t>(atoms)};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<uint8_t*>(wq), dims, strides,
                          box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MXFP4_OK : MXFP4_ERR_CUDA;
}

// Packed weights [rows, k/2] for the packed-E2M1 tensor-core kernel: the 3D
// view (128 B, rows, k/256) with strides (k/2 B, 128 B) and a box of 2
// atoms x box_rows rows, so one copy lands [atom][row][128 B] swizzled, the
// codes as stored. Needs k % 512 == 0.
int encode_f4_weight_map(CUtensorMap* map, const uint8_t* wq, int64_t rows, int64_t k, int box_rows) {
    cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(k / 256)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(k / 2), 128};
    cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), 2};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(wq), dims, strides, box,
                          estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MXFP4_OK : MXFP4_ERR_CUDA;
}

}  // namespace

namespace mxfp4 {
int encode_weights(CUtensorMap* map, const uint8_t* wq, int64_t rows, int64_t k, int steps, int* is3d) {
    return encode_weight_map(map, wq, rows, k, steps, is3d);
}

// One copy per stage for units whose boxes are consecutive 16-row groups:
// the 3D view with a box of box_rows rows (mode 2 of the engine). Falls back
// to encode_weights (mode 0) when k % 256 != 0.
int encode_weights_merged_rows(CUtensorMap* map, const uint8_t* wq, int64_t rows, int64_t k, int steps, int box_rows,
                               int* mode) {
    if (k % 256 == 0) {
        cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(k / 256)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(k / 2), 128};
        cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(steps)};
        cuuint32_t estride[3] = {1, 1, 1};
        const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(wq), dims, strides, box,
                                    estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r == CUDA_SUCCESS) {
            *mode = 2;
            return MXFP4_OK;
        }
    }
    int is3d = 0;
    const int rc = encode_weight_map(map, wq, rows, k, steps, &is3d);
    *mode = is3d;
    return rc;
}

// One copy per stage for gate/up units of W1 [e][2*inter][k/2] (16 gate rows
// and the 16 up rows inter rows below them): the 5D view (128 B, 16 rows,
// gate/up, 16-row group, k/256) with strides (k/2, inter*k/2, 16*k/2, 128 B)
// and a box of one group's gate and up rows (mode 3 of the engine). A unit
// starting at row r (a gate row, r % 16 == 0) is group r / 16. Falls back to
// encode_weights (mode 0) when k % 256 != 0.
int encode_weights_gate_up(CUtensorMap* map, const uint8_t* w1q, int64_t experts, int64_t inter, int64_t k, int steps,
                           int* mode) {
    if (k % 256 == 0 && inter % 16 == 0) {
        cuuint64_t dims[5] = {128, 16, 2, static_cast<cuuint64_t>(experts * inter / 8), static_cast<cuuint64_t>(k / 256)};
        cuuint64_t strides[4] = {static_cast<cuuint64_t>(k / 2), static_cast<cuuint64_t>(inter * (k / 2)),
                                 static_cast<cuuint64_t>(16 * (k / 2)), 128};
        cuuint32_t box[5] = {128, 16, 2, 1, static_cast<cuuint32_t>(steps)};
        cuuint32_t estride[5] = {1, 1, 1, 1, 1};
        const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<uint8_t*>(w1q), dims, strides,
                                    box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r == CUDA_SUCCESS) {
            *mode = 3;
            return MXFP4_OK;
        }
    }
    int is3d = 0;
    const int rc = encode_weight_map(map, w1q, experts * 2 * inter, k, steps, &is3d);
    *mode = is3d;
    return rc;
}
}  // namespace mxfp4

namespace {

// Plans and TMA descriptors of recent linear calls, per host thread: a
// layer calls with the same weights and shape every step, and the plan and
// the descriptor (which embeds the weight address) depend on nothing else.
struct LinearPlan {
    int dev = -1;
    const uint8_t* wq = nullptr;
    const uint8_t* ws = nullptr;
    int64_t t = 0, k = 0, n = 0;
    int kind = 0;  // 0: streaming engine; 1: E4M3-split tensor-core kernel; 2: packed-E2M1 tensor-core kernel
    mxfp4::LinearParams p{};
    mxfp4::tc::TcPlan tp{};
    mxfp4::f4::F4Plan fp{};
    CUtensorMap map;
    CUtensorMap tail_map;  // kind 2 with a tail tile
};
constexpr int kPlanCache = 16;
thread_local LinearPlan t_plans[kPlanCache];
thread_local int t_plan_next = 0;

// The launch plan of a linear call (host only): cluster size and shared
// memory layout for t tokens, k, n on a device with num_sms SMs and max_smem
// bytes of opt-in shared memory per block. False if no plan fits.
bool linear_plan(int64_t t, int64_t k, int64_t n, int num_sms, int max_smem, int* cl, mxfp4::SmemLayout* L) {
    const int64_t n_rg = (n + 15) / 16;
    const bool few_units = n_rg <= 4 * static_cast<int64_t>(num_sms);
    const int64_t ctas = n_rg < num_sms ? n_rg : num_sms;
    const int units_per_cta = static_cast<int>((n_rg + ctas - 1) / ctas);
    return mxfp4::plan_linear(static_cast<int>(t), static_cast<int>(k), max_smem, few_units, units_per_cta, cl, L);
}

// Argument checks shared by mxfp4_linear and mxfp4_linear_plan.
int linear_shape_status(int64_t t, int64_t k, int64_t n) {
    if (t <= 0 || k <= 0 || n <= 0) return MXFP4_ERR_INVALID_ARG;
    if (k % 32 != 0 || t > 32 || n >= (int64_t(1) << 31) || k >= (int64_t(1) << 31)) return MXFP4_ERR_SHAPE;
    return MXFP4_OK;
}

// Kernel arguments of one packed-E2M1 call with plan fp (inputs and outputs
// set by the caller).
mxfp4::f4::F4Params f4_params(const mxfp4::f4::F4Plan& fp, const uint8_t* ws, unsigned* status, int64_t t,
                              int64_t k, int64_t n) {
    mxfp4::f4::F4Params q{};
    q.ws = ws;
    q.status = status;
    q.T = static_cast<int>(t);
    q.K = static_cast<int>(k);
    q.N = static_cast<int>(n);
    q.nblk = static_cast<int>(k / 32);
    q.stages = static_cast<int>(k / 512);
    q.rows = fp.rows;
    q.h_main = fp.h_main;
    q.h_tail = fp.h_tail;
    q.cl = fp.cl;
    q.na = fp.na;
    q.nb = fp.nb;
    q.max_batch = fp.max_batch;
    q.tmem_cols = fp.tmem_cols;
    q.inbox_bytes = fp.inbox_bytes;
    return q;
}

// The FFN chain on the packed-E2M1 kernel: W1 [2 inter, hidden] with fp32
// outputs a | b into the workspace, then W2 [hidden, inter] whose
// conversion takes SiLU(a) * b. Plans and tensor maps per weight set.
struct FfnF4Plan {
    int dev = -1;
    const uint8_t* w1q = nullptr;
    const uint8_t* w2q = nullptr;
    int64_t t = 0, hidden = 0, inter = 0;
    mxfp4::f4::F4Plan up{}, down{};
    CUtensorMap up_map, up_tail, down_map, down_tail;
};
thread_local FfnF4Plan t_ffn_plans[4];
thread_local int t_ffn_next = 0;

// The plan of an FFN call on the packed-E2M1 kernel, or null when the shape
// is outside it (t > 4, hidden or inter not a multiple of 512, no fit).
const FfnF4Plan* ffn_f4_plan(int dev, const DeviceInfo* d, const uint8_t* w1q, const uint8_t* w2q, int64_t t,
                             int64_t hidden, int64_t inter, int* rc) {
    *rc = MXFP4_OK;
    for (const FfnF4Plan& c : t_ffn_plans)
        if (c.dev == dev && c.w1q == w1q && c.w2q == w2q && c.t == t && c.hidden == hidden && c.inter == inter)
            return &c;
    if (t > 4 || hidden % 512 != 0 || inter % 512 != 0) return nullptr;
    FfnF4Plan f;
    if (!mxfp4::f4::plan_f4(static_cast<int>(t), hidden, 2 * inter, d->num_sms, d->max_smem, &f.up) ||
        !mxfp4::f4::plan_f4(static_cast<int>(t), inter, hidden, d->num_sms, d->max_smem, &f.down, true))
        return nullptr;
    if ((*rc = encode_f4_weight_map(&f.up_map, w1q, 2 * inter, hidden, f.up.h_main))) return nullptr;
    f.up_tail = f.up_map;
    if (f.up.h_tail && (*rc = encode_f4_weight_map(&f.up_tail, w1q, 2 * inter, hidden, f.up.h_tail))) return nullptr;
    if ((*rc = encode_f4_weight_map(&f.down_map, w2q, hidden, inter, f.down.h_main))) return nullptr;
    f.down_tail = f.down_map;
    if (f.down.h_tail && (*rc = encode_f4_weight_map(&f.down_tail, w2q, hidden, inter, f.down.h_tail)))
        return nullptr;
    f.dev = dev;
    f.w1q = w1q;
    f.w2q = w2q;
    f.t = t;
    f.hidden = hidden;
    f.inter = inter;
    FfnF4Plan* slot = &t_ffn_plans[t_ffn_next];
    t_ffn_next = (t_ffn_next + 1) % 4;
    *slot = f;
    return slot;
}

}  // namespace

extern "C" {

const char* mxfp4_strerror(int status) {
    switch (status) {
        case MXFP4_OK: return "MXFP4_OK";
        case MXFP4_ERR_INVALID_ARG: return "MXFP4_ERR_INVALID_ARG: null pointer or non-positive size";
        case MXFP4_ERR_SHAPE: return "MXFP4_ERR_SHAPE: unsupported size";
        case MXFP4_ERR_ALIGN: return "MXFP4_ERR_ALIGN: pointer not aligned as documented";
        case MXFP4_ERR_WORKSPACE: return "MXFP4_ERR_WORKSPACE: workspace missing or too small";
        case MXFP4_ERR_CUDA: return "MXFP4_ERR_CUDA: CUDA runtime or launch failure";
        case MXFP4_ERR_TIMEOUT: return "MXFP4_ERR_TIMEOUT: a device-side bounded wait expired";
        default: return "MXFP4: unknown status";
    }
}

int mxfp4_quantize(const float* w, int64_t n, int64_t k, uint8_t* wq, uint8_t* ws, void* stream) {
    if (!w || !wq || !ws || n <= 0 || k <= 0) return MXFP4_ERR_INVALID_ARG;
    if (k % 32 != 0) return MXFP4_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(wq, 16)) return MXFP4_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    if (int rc = device_info(&d)) return rc;
    cudaError_t e = mxfp4::launch_quantize(w, n, k, wq, ws, static_cast<cudaStream_t>(stream), d->num_sms);
    return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}

int mxfp4_linear(const void* x, int64_t t, int64_t k, const uint8_t* wq, const uint8_t* ws, int64_t n, void* y,
                 void* stream) {
    if (!x || !wq || !ws || !y) return MXFP4_ERR_INVALID_ARG;
    if (int rc = linear_shape_status(t, k, n)) return rc;
    if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(ws, 16) || !aligned(y, 2)) return MXFP4_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    if (int rc = device_info(&d)) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    LinearPlan* plan = nullptr;
    for (LinearPlan& c : t_plans)
        if (c.dev == dev && c.wq == wq && c.ws == ws && c.t == t && c.k == k && c.n == n) {
            plan = &c;
            break;
        }
    if (!plan) {
        LinearPlan fresh;
        // The packed-E2M1 tensor-core kernel when its plan fits (k % 512 ==
        // 0; t <= 8, or t <= 16 with one batch per CTA). Then the E4M3-split
        // tensor-core kernel when the shape and the weight alignment allow
        // it; the streaming engine otherwise.
        if (mxfp4::f4::plan_f4(static_cast<int>(t), k, n, d->num_sms, d->max_smem, &fresh.fp)) {
            fresh.kind = 2;
            if (int rc = encode_f4_weight_map(&fresh.map, wq, n, k, fresh.fp.h_main)) return rc;
            fresh.tail_map = fresh.map;
            if (fresh.fp.h_tail)
                if (int rc = encode_f4_weight_map(&fresh.tail_map, wq, n, k, fresh.fp.h_tail)) return rc;
        } else if (aligned(wq, 32) &&
                   mxfp4::tc::plan_tc(static_cast<int>(t), k, n, d->num_sms, d->max_smem, &fresh.tp)) {
            fresh.kind = 1;
            if (int rc = encode_tc_weight_map(&fresh.map, wq, n, k, fresh.tp.atoms_per_stage)) return rc;
        } else {
            if (!linear_plan(t, k, n, d->num_sms, d->max_smem, &fresh.p.cl, &fresh.p.layout)) return MXFP4_ERR_SHAPE;
            if (int rc =
                    encode_weight_map(&fresh.map, wq, n, k, static_cast<int>(fresh.p.layout.steps), &fresh.p.tma3d))
                return rc;
        }
        fresh.dev = dev;
        fresh.wq = wq;
        fresh.ws = ws;
        fresh.t = t;
        fresh.k = k;
        fresh.n = n;
        plan = &t_plans[t_plan_next];
        t_plan_next = (t_plan_next + 1) % kPlanCache;
        *plan = fresh;
    }
    const CUtensorMap& map = plan->map;
    if (plan->kind == 2) {
        const mxfp4::f4::F4Plan& fp = plan->fp;
        mxfp4::f4::F4Params q = f4_params(fp, ws, d->status, t, k, n);
        q.x = static_cast<const __nv_bfloat16*>(x);
        q.y = static_cast<__nv_bfloat16*>(y);
        cudaError_t e = mxfp4::f4::launch_f4_linear(map, plan->tail_map, q, fp, static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
    }
    if (plan->kind == 1) {
        mxfp4::tc::TcLinearParams q{};
        q.x = static_cast<const __nv_bfloat16*>(x);
        q.ws = ws;
        q.y = static_cast<__nv_bfloat16*>(y);
        q.status = d->status;
        q.T = static_cast<int>(t);
        q.K = static_cast<int>(k);
        q.N = static_cast<int>(n);
        q.nblk = static_cast<int>(k / 32);
        q.stages = plan->tp.stages;
        q.tiles = plan->tp.tiles;
        q.cl = plan->tp.cl;
        cudaError_t e = mxfp4::tc::launch_tc_linear(map, q, plan->tp, static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
    }
    mxfp4::LinearParams p = plan->p;
    p.x = static_cast<const __nv_bfloat16*>(x);
    p.ws = ws;
    p.y = static_cast<__nv_bfloat16*>(y);
    p.status = d->status;
    p.T = static_cast<int>(t);
    p.K = static_cast<int>(k);
    p.N = static_cast<int>(n);
    p.nblk = static_cast<int>(k / 32);
    p.nkb = static_cast<int>((k + 255) / 256);
    p.xcols = static_cast<int>(t);
    p.n_rg = static_cast<int>((n + 15) / 16);
    cudaError_t e = mxfp4::launch_linear(map, p, d->num_sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}

int mxfp4_linear_plan(int64_t t, int64_t k, int64_t n, int num_sms, int max_smem, mxfp4_linear_plan_t* out) {
    if (!out || num_sms <= 0 || max_smem <= 0) return MXFP4_ERR_INVALID_ARG;
    if (int rc = linear_shape_status(t, k, n)) return rc;
    mxfp4::f4::F4Plan fp{};
    if (mxfp4::f4::plan_f4(static_cast<int>(t), k, n, num_sms, max_smem, &fp)) {
        mxfp4_linear_plan_t r{};
        r.mode = 4;
        r.ctas = fp.grid;
        r.cluster = fp.cl;
        r.stage_steps = 2;  // 512 K values per stage
        r.chunk_steps = 2;
        r.ring_slots = fp.na;
        r.part_steps = 0;
        r.batch_units = fp.tiles;  // tiles of at most 128 rows per group
        r.smem_bytes = fp.smem_bytes;
        r.group_rows = fp.rows;
        *out = r;
        return MXFP4_OK;
    }
    mxfp4::tc::TcPlan tp{};
    if (mxfp4::tc::plan_tc(static_cast<int>(t), k, n, num_sms, max_smem, &tp)) {
        mxfp4_linear_plan_t r{};
        r.mode = 3;
        r.ctas = tp.grid;
        r.cluster = tp.cl;
        r.stage_steps = tp.atoms_per_stage / 2;  // 128-value atoms -> 256-value steps
        r.chunk_steps = r.stage_steps;
        r.ring_slots = tp.ring_slots;
        r.part_steps = 0;
        r.batch_units = (tp.tiles + tp.grid / tp.cl - 1) / (tp.grid / tp.cl);  // 128-row tiles per CTA (at most)
        r.smem_bytes = tp.smem_bytes;
        *out = r;
        return MXFP4_OK;
    }
    int cl = 1;
    mxfp4::SmemLayout L{};
    if (!linear_plan(t, k, n, num_sms, max_smem, &cl, &L)) return MXFP4_ERR_SHAPE;
    const int64_t n_rg = (n + 15) / 16;
    mxfp4_linear_plan_t r{};
    r.mode = L.part_steps ? 1 : (cl > 1 ? 2 : 0);
    r.cluster = cl;
    // CTAs: one per SM, never more groups than row groups; for clusters the
    // co-resident cluster count at launch may be lower than this bound.
    const int64_t groups = cl > 1 ? num_sms / cl : num_sms;
    r.ctas = static_cast<int32_t>(cl * (groups < n_rg ? groups : n_rg));
    r.stage_steps = static_cast<int32_t>(L.steps);
    r.chunk_steps = static_cast<int32_t>(L.group);
    r.ring_slots = static_cast<int32_t>(L.nslot);
    r.part_steps = static_cast<int32_t>(L.part_steps);
    r.batch_units = static_cast<int32_t>(L.ubatch);
    r.smem_bytes = static_cast<int32_t>(L.total) + 1024;  // + alignment slack, as launched
    *out = r;
    return MXFP4_OK;
}

size_t mxfp4_moe_workspace_size(int64_t t, int64_t e, int top_k, int64_t hidden, int64_t inter) {
    if (t <= 0 || e <= 0 || top_k <= 0 || hidden <= 0 || inter <= 0) return 0;
    return mxfp4::moe_workspace_bytes(t, e, top_k, hidden, inter);
}

size_t mxfp4_moe_shared_workspace_size(int64_t t, int64_t e, int top_k, int n_shared, int64_t hidden,
                                       int64_t inter) {
    if (t <= 0 || e <= 0 || top_k <= 0 || n_shared < 0 || hidden <= 0 || inter <= 0) return 0;
    return mxfp4::moe_workspace_bytes(t, e, top_k + n_shared, hidden, inter);
}

}  // extern "C"

namespace {

int moe_call(const void* x, int64_t t, int64_t hidden, const float* router_logits, int64_t e, int top_k,
             int n_shared, const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q, const uint8_t* w2s,
             int64_t inter, void* y, int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes,
             void* stream) {
    if (!x || !router_logits || !w1q || !w1s || !w2q || !w2s || !y || t <= 0 || hidden <= 0 || e <= 0 ||
        top_k <= 0 || inter <= 0 || n_shared < 0)
        return MXFP4_ERR_INVALID_ARG;
    const int64_t et = e + n_shared;  // experts in the weight arrays
    if (hidden % 32 != 0 || inter % 32 != 0 || t > 256 || e > 1024 || top_k > 16 || top_k > e ||
        n_shared > 16 || et > 1024)
        return MXFP4_ERR_SHAPE;
    if (et * 2 * inter >= (int64_t(1) << 31) || et * hidden >= (int64_t(1) << 31)) return MXFP4_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(w1q, 16) || !aligned(w1s, 16) || !aligned(w2q, 16) || !aligned(w2s, 16) ||
        !aligned(y, 2) || !aligned(router_logits, 4) || (topk_ids && !aligned(topk_ids, 4)) ||
        (topk_w && !aligned(topk_w, 4)))
        return MXFP4_ERR_ALIGN;
    if (!workspace) return MXFP4_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return MXFP4_ERR_ALIGN;
    if (workspace_bytes < mxfp4::moe_workspace_bytes(t, e, top_k + n_shared, hidden, inter))
        return MXFP4_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    if (int rc = device_info(&d)) return rc;
    mxfp4::MoeArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.logits = router_logits;
    a.w1q = w1q;
    a.w1s = w1s;
    a.w2q = w2q;
    a.w2s = w2s;
    a.y = static_cast<__nv_bfloat16*>(y);
    a.topk_ids = topk_ids;
    a.topk_w = topk_w;
    a.workspace = workspace;
    a.status = d->status;
    a.T = static_cast<int>(t);
    a.E = static_cast<int>(e);
    a.top_k = top_k;
    a.hidden = static_cast<int>(hidden);
    a.inter = static_cast<int>(inter);
    a.n_shared = n_shared;
    return mxfp4::launch_moe(w1q, w2q, a, d->num_sms, d->max_smem, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int mxfp4_moe(const void* x, int64_t t, int64_t hidden, const float* router_logits, int64_t e, int top_k,
              const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q, const uint8_t* w2s, int64_t inter, void* y,
              int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes, void* stream) {
    return moe_call(x, t, hidden, router_logits, e, top_k, 0, w1q, w1s, w2q, w2s, inter, y, topk_ids, topk_w,
                    workspace, workspace_bytes, stream);
}

int mxfp4_moe_shared(const void* x, int64_t t, int64_t hidden, const float* router_logits, int64_t e, int top_k,
                     int n_shared, const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q, const uint8_t* w2s,
                     int64_t inter, void* y, int32_t* topk_ids, float* topk_w, void* workspace,
                     size_t workspace_bytes, void* stream) {
    return moe_call(x, t, hidden, router_logits, e, top_k, n_shared, w1q, w1s, w2q, w2s, inter, y, topk_ids,
                    topk_w, workspace, workspace_bytes, stream);
}

size_t mxfp4_ffn_workspace_size(int64_t t, int64_t hidden, int64_t inter) {
    if (t <= 0 || hidden <= 0 || inter <= 0) return 0;
    return mxfp4::ffn_workspace_bytes(t, inter);
}

int mxfp4_ffn(const void* x, int64_t t, int64_t hidden, const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q,
              const uint8_t* w2s, int64_t inter, void* y, void* workspace, size_t workspace_bytes, void* stream) {
    if (!x || !w1q || !w1s || !w2q || !w2s || !y || t <= 0 || hidden <= 0 || inter <= 0)
        return MXFP4_ERR_INVALID_ARG;
    if (t > 8 || hidden % 32 != 0 || inter % 32 != 0 || hidden > (1 << 20) || inter > (1 << 20))
        return MXFP4_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(w1q, 16) || !aligned(w1s, 16) || !aligned(w2q, 16) || !aligned(w2s, 16) ||
        !aligned(y, 2))
        return MXFP4_ERR_ALIGN;
    if (!workspace) return MXFP4_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return MXFP4_ERR_ALIGN;
    if (workspace_bytes < mxfp4::ffn_workspace_bytes(t, inter)) return MXFP4_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    if (int rc = device_info(&d)) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    int prc = MXFP4_OK;
    if (const FfnF4Plan* f = ffn_f4_plan(dev, d, w1q, w2q, t, hidden, inter, &prc)) {
        // Two launches on the stream, the second waiting for the first only
        // where it reads a | b (programmatic dependent launch).
        float* ab = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 256);
        mxfp4::f4::F4Params q1 = f4_params(f->up, w1s, d->status, t, hidden, 2 * inter);
        q1.x = static_cast<const __nv_bfloat16*>(x);
        q1.yf = ab;
        cudaError_t e = mxfp4::f4::launch_f4_linear(f->up_map, f->up_tail, q1, f->up, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return MXFP4_ERR_CUDA;
        mxfp4::f4::F4Params q2 = f4_params(f->down, w2s, d->status, t, inter, hidden);
        q2.xab = ab;
        q2.y = static_cast<__nv_bfloat16*>(y);
        e = mxfp4::f4::launch_f4_linear(f->down_map, f->down_tail, q2, f->down, static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
    }
    if (prc != MXFP4_OK) return prc;
    mxfp4::FfnPlan plan{};
    if (int rc = mxfp4::plan_ffn(static_cast<int>(t), static_cast<int>(hidden), static_cast<int>(inter), d->max_smem,
                                 &plan))
        return rc;
    mxfp4::FfnArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.w1q = w1q;
    a.w1s = w1s;
    a.w2q = w2q;
    a.w2s = w2s;
    a.y = static_cast<__nv_bfloat16*>(y);
    a.workspace = workspace;
    a.status = d->status;
    a.T = static_cast<int>(t);
    a.hidden = static_cast<int>(hidden);
    a.inter = static_cast<int>(inter);
    return mxfp4::launch_ffn(a, d->num_sms, d->max_smem, static_cast<cudaStream_t>(stream));
}

int mxfp4_last_device_status(void* stream) {
    DeviceInfo* d = nullptr;
    if (int rc = device_info(&d)) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MXFP4_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof word) != cudaSuccess) return MXFP4_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess) return MXFP4_ERR_CUDA;
    return (word & mxfp4::kStatusTimeout) ? MXFP4_ERR_TIMEOUT : MXFP4_OK;
}

}  // extern "C"
