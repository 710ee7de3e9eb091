// fg_gemm_nt.cu - NT (K-major A and B) kernel variants: dense, M-grouped contiguous and
// M-grouped masked GEMMs.
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<64, false>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, false>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<192, false>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, false>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, false>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
// CTA-pair variants (dense)
template cudaError_t launch_gemm<128, false, true>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, false, true>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, false, true>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t max_active_clusters<128, false, true>(int, int*);
template cudaError_t max_active_clusters<224, false, true>(int, int*);
template cudaError_t max_active_clusters<256, false, true>(int, int*);
}  // namespace fg
