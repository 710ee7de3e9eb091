// fg_gemm_swiglu.cu - the gate-up GEMM with the fused SwiGLU + per-1x128 FP8
// requantisation epilogue (NT, 256-row B tiles of 128 gate + 128 up rows), with E4M3
// weights (128x128-block scales) or packed E2M1 weights (one scale per 32 K elements of a
// row), compiled in its own translation unit.
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<256, kMajNT, false, true, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajNT, false, true, false, kMasked>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajNTF4, false, true, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajNTF4, false, true, false, kMasked>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
}  // namespace fg
