// fg_gemm_nt.cu - NT (K-major A and B) kernel variants of the M-grouped contiguous and
// M-grouped masked GEMMs (one variant per layout: the tile walk is fixed at compile time).
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<64, kMajNT, false, false, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNT, false, false, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<192, kMajNT, false, false, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajNT, false, false, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajNT, false, false, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<64, kMajNT, false, false, false, kMasked>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNT, false, false, false, kMasked>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<192, kMajNT, false, false, false, kMasked>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajNT, false, false, false, kMasked>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<256, kMajNT, false, false, false, kMasked>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
}  // namespace fg
