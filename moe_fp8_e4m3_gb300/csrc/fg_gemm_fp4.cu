// fg_gemm_fp4.cu - FP8 x FP4 kernel variants (A E4M3 with 1x128 scales, B packed E2M1 with
// one scale per 32 K elements of a row): dense NT at tile widths 128 and 224 (with and
// without C slots), dense split-K clusters at 128, M-grouped contiguous and masked at 128
// and 224.
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<128, kMajNTF4, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajNTF4, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNTF4, false, false, true, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajNTF4, false, false, true, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNTF4, true, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
}  // namespace fg
