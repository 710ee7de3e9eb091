// fg_gemm_split.cu - split-K cluster variants of the dense NT kernel (one tile per
// cluster, partial tiles summed through distributed shared memory), compiled in their
// own translation unit.
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<64, kMajNT, true, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNT, true, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<192, kMajNT, true, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajNT, true, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajNT, true, false, false, kDense>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t max_active_clusters<64, kMajNT, true, false, false, kDense>(int, int*);
template cudaError_t max_active_clusters<128, kMajNT, true, false, false, kDense>(int, int*);
template cudaError_t max_active_clusters<192, kMajNT, true, false, false, kDense>(int, int*);
template cudaError_t max_active_clusters<224, kMajNT, true, false, false, kDense>(int, int*);
template cudaError_t max_active_clusters<256, kMajNT, true, false, false, kDense>(int, int*);
}  // namespace fg
