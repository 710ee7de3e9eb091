// fg_gemm_tn.cu - TN (MN-major A and B) kernel variants: the K-grouped weight-gradient GEMM.
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<128, kMajTN>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajTN>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
}  // namespace fg
