// Test-only pin: exposes CUDA's host-side FP4/E8M0 conversions from
// cuda_fp4.h / cuda_fp8.h (library routines, compiled here with g++ for the
// host) so the oracle's decode table, E8M0 decode and E2M1 rounding can be
// checked against an implementation that is not the oracle's.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

extern "C" {

float pin_e2m1_decode(int code) {
    __nv_fp4_e2m1 v;
    v.__x = (__nv_fp4_storage_t)(code & 15);
    return (float)v;
}

// Round a double to E2M1 (round to nearest even, saturating to finite).
int pin_e2m1_round(double v) {
    return (int)__nv_cvt_double_to_fp4(v, __NV_E2M1, cudaRoundNearest) & 15;
}

float pin_e8m0_decode(int s) {
    __nv_fp8_e8m0 v;
    v.__x = (__nv_fp8_storage_t)s;
    return (float)v;
}

}
