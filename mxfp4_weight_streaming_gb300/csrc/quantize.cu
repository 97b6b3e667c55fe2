// MXFP4 packer for sm_103a: one thread per 32-value block.
//
// Format ("Zyphra Inference Wave 2", section "Quantization"): each block of
// 32 values shares one E8M0 power-of-two scale; each value is an E2M1 code.
// Scale rule (OCP MX): s = clamp(floor(log2 amax) - 2 + 127, 0, 254), with
// floor(log2) read from the float32 exponent bits (or the leading mantissa
// bit of a subnormal). Each value is multiplied by 2^(127-s), which is exact
// here, and rounded by the hardware float32 -> E2M1 conversion (round to
// nearest even, saturating to +-6, sign kept).
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"

namespace mxfp4 {

__device__ __forceinline__ uint32_t pack_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u32.u8 %0, b;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(256) quantize_kernel(const float* __restrict__ w, int64_t nblocks,
                                                       uint8_t* __restrict__ wq, uint8_t* __restrict__ ws) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblocks;
         i += (int64_t)gridDim.x * blockDim.x) {
        // Rows are K-contiguous and K % 32 == 0, so block i starts at w + 32 i.
        const float4* src = reinterpret_cast<const float4*>(w + i * 32);
        float v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float4 f = __ldg(src + q);
            v[4 * q] = f.x;
            v[4 * q + 1] = f.y;
            v[4 * q + 2] = f.z;
            v[4 * q + 3] = f.w;
        }
        uint32_t amax_bits = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax_bits = max(amax_bits, __float_as_uint(v[j]) & 0x7fffffffu);
        int s = 0;
        if (amax_bits != 0) {
            const int biased = static_cast<int>(amax_bits >> 23);
            const int fl = biased ? biased - 127 : (31 - __clz(static_cast<int>(amax_bits))) - 149;
            s = min(254, max(0, fl - 2 + 127));
        }
        const float inv = exp2_int(127 - s);  // 127 - s in [-127, 127]
        uint32_t out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = 8 * q + 2 * j;
                word |= pack_e2m1x2(v[e] * inv, v[e + 1] * inv) << (8 * j);
            }
            out[q] = word;
        }
        reinterpret_cast<uint4*>(wq)[i] = make_uint4(out[0], out[1], out[2], out[3]);
        ws[i] = static_cast<uint8_t>(s);
    }
}

cudaError_t launch_quantize(const float* w, int64_t n, int64_t k, uint8_t* wq, uint8_t* ws, cudaStream_t stream,
                            int num_sms) {
    const int64_t nblocks = n * (k / 32);
    const int threads = 256;
    int64_t grid = (nblocks + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (grid > cap) grid = cap;
    quantize_kernel<<<static_cast<unsigned>(grid), threads, 0, stream>>>(w, nblocks, wq, ws);
    return cudaGetLastError();
}

}  // namespace mxfp4
