// fg_launch.h - host-side declarations shared by the C-ABI layer and the kernel
// instantiation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fg_gemm_kernel.cuh"

namespace fg {

// Launches fg_gemm_kernel<BN, kTN> with `grid` persistent CTAs on `stream`.
template <int BN, bool kTN>
cudaError_t launch_gemm(const GemmParams& p, const CUtensorMap& map_a, const CUtensorMap& map_b,
                        const CUtensorMap& map_c, const CUtensorMap& map_d, int grid, cudaStream_t stream);

}  // namespace fg
