// fg_gemm_tn.cu - TN (MN-major A and B) kernel variants: the dense TN GEMM and the
// K-grouped weight-gradient GEMM.
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<128, kMajTN, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajTN, false, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajTN, false, false, false, kKGrouped>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajTN, false, false, false, kKGrouped>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
}  // namespace fg
