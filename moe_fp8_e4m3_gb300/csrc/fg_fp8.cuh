// fg_fp8.cuh - the activation quantisation rule shared by the quantise kernels and the
// GEMM's fused SwiGLU epilogue: per group, the smallest power-of-two scale 2^e with
// amax <= 448 * 2^e (UE8M0 byte e + 127, clamped to [0, 254]; an all-zero group gets
// byte 127), and codes E4M3 round-to-nearest-even of x * 2^-e.
#pragma once

#include <cuda_fp8.h>
#include <cstdint>

namespace fg {

__device__ __forceinline__ int scale_exponent(float amax) {
    if (!(amax > 0.0f)) return 0;
    int ex;
    const float fr = frexpf(amax, &ex);     // amax = fr * 2^ex, fr in [0.5, 1)
    // amax / 2^(ex-9) = 512 fr lies in [256, 512): within 448 iff fr <= 0.875
    int e = fr <= 0.875f ? ex - 9 : ex - 8;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    return e;
}

__device__ __forceinline__ uint32_t e4m3(float v) {
    return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

}  // namespace fg
