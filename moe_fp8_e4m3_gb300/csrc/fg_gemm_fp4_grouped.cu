// fg_gemm_fp4_grouped.cu - FP8 x FP4 kernel variants of the M-grouped contiguous and masked
// GEMMs (B packed E2M1 with one scale per 32 K elements of a row) at tile widths 128 and 224.
#include "fg_gemm_inst.cuh"

namespace fg {
template cudaError_t launch_gemm<128, kMajNTF4, false, false, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajNTF4, false, false, false, kContiguous>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<128, kMajNTF4, false, false, false, kMasked>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
template cudaError_t launch_gemm<224, kMajNTF4, false, false, false, kMasked>(const GemmParams&, const GemmMaps&, int, cudaStream_t);
}  // namespace fg
