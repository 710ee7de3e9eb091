// fg_gemm_nt.cu - NT (K-major A and B) kernel variants: dense, M-grouped contiguous and
// M-grouped masked GEMMs.
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<64, kMajNT>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNT>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<192, kMajNT>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajNT>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajNT>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
}  // namespace fg
