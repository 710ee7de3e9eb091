// fg_gemm_layouts.cu - variants with an N-major B ([K][N]: dense NN and M-grouped contiguous
// NN) or an M-major A ([K][M]: dense TT), compiled in their own translation unit.  The
// TN variants (both operands MN-major) are in fg_gemm_tn.cu.
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<128, kMajNN, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajNN, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNN, false, false, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajNN, false, false, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajTT, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajTT, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajTT, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
}  // namespace fg
