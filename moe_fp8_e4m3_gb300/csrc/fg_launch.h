// fg_launch.h - host-side declarations shared by the C-ABI layer and the kernel
// instantiation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fg_gemm_kernel.cuh"

namespace fg {

// Launches fg_gemm_kernel<BN, kMaj, kSplit, kSwiGLU, kSepC, kKindT> with `grid` persistent CTAs on `stream`.
// kMaj: operand majors (kMajNT, kMajNN, kMajTN, kMajTT).
// kSplit: clusters of p.split CTAs sharing one tile along K (dense NT only).
// kSwiGLU: BN = 256 tiles of 128 gate + 128 up columns, SwiGLU + FP8 requantisation epilogue.
// kSepC: shared-memory slots that prefetch C, for a C that is not D (fewer pipeline stages).
// kKindT: the layout (GemmKind) the variant serves, fixed at compile time (-1: read from p.kind).
template <int BN, int kMaj, bool kSplit = false, bool kSwiGLU = false, bool kSepC = false, int kKindT = -1>
cudaError_t launch_gemm(const GemmParams& p, const GemmMaps& maps, int grid, cudaStream_t stream);

// How many clusters of `cluster` CTAs of fg_gemm_kernel<BN, kMaj, kSplit, kSwiGLU, kSepC, kKindT> can be resident at once.
template <int BN, int kMaj, bool kSplit = false, bool kSwiGLU = false, bool kSepC = false, int kKindT = -1>
cudaError_t max_active_clusters(int cluster, int* out);

}  // namespace fg
