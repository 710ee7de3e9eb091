// fg_gemm_sepc.cu - the variants with C prefetch slots, launched when C is an array of its
// own (not D): every tile width that has two accumulators, in the layouts that take C
// (dense NT, NN, TT; dense and K-grouped TN).
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<64, kMajNT, false, false, true, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNT, false, false, true, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<192, kMajNT, false, false, true, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajNT, false, false, true, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajTN, false, false, true, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajTN, false, false, true, kKGrouped>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNN, false, false, true, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajTT, false, false, true, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajTT, false, false, true, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
}  // namespace fg
