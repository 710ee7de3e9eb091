// fg_gemm_inst.cuh - definition of launch_gemm, included by the instantiation units so
// that the kernel variants compile in parallel translation units.
#pragma once

#include <mutex>

#include "fg_launch.h"

namespace fg {

template <int BN, bool kTN, bool k2Sm>
cudaError_t launch_gemm(const GemmParams& p, const CUtensorMap& map_a, const CUtensorMap& map_b,
                        const CUtensorMap& map_c, const CUtensorMap& map_d, int grid, cudaStream_t stream) {
    constexpr int kSmem = TileCfg<BN, k2Sm>::kSmemBytes;
    auto kernel = fg_gemm_kernel<BN, kTN, k2Sm>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    static std::mutex mu;
    static bool configured[256] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
        if (!configured[dev]) {
            err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
            if (err != cudaSuccess) return err;
            configured[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(224);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (k2Sm) {   // CTA pairs: grid is even, clusters of two along x
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, p, map_a, map_b, map_c, map_d);
}

}  // namespace fg
