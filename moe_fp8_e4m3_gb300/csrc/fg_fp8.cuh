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

// 2^-e as a float, built from its exponent bits: an exact multiplier for e in [-127, 126]
// (a finite amax gives e <= 120; the clamp only keeps the bits valid).  x * 2^-e equals
// the scaling x / 2^e exactly wherever the result is a normal float.
__device__ __forceinline__ float pow2_neg(int e) {
    e = e > 126 ? 126 : e;
    return __int_as_float((127 - e) << 23);
}

// Four already-scaled values to E4M3 (saturating, round to nearest even) in one word, the
// first in the low byte; the values go through the paired conversion two at a time.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xFFFFu) | (hi & 0xFFFFu) << 16;
}

}  // namespace fg
