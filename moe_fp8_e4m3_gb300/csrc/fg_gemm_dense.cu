// fg_gemm_dense.cu - the dense NT variants without split or C slots.
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<64, kMajNT, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNT, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<192, kMajNT, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajNT, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajNT, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
}  // namespace fg
