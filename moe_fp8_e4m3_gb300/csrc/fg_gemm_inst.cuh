// fg_gemm_inst.cuh - definition of launch_gemm, included by the instantiation units so
// that the kernel variants compile in parallel translation units.
#pragma once

#include <mutex>

#include "fg_launch.h"

namespace fg {

// Raises the kernel's dynamic shared-memory limit once per device.
template <int BN, int kMaj, bool kSplit, bool kSwiGLU, bool kSepC, int kKindT>
cudaError_t configure_gemm() {
    constexpr int kSmem = TileCfg<BN, kSplit, kSwiGLU, kSepC>::kSmemBytes;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    static std::mutex mu;
    static bool configured[256] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        err = cudaFuncSetAttribute(fg_gemm_kernel<BN, kMaj, kSplit, kSwiGLU, kSepC, kKindT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (err != cudaSuccess) return err;
        configured[dev] = true;
    }
    return cudaSuccess;
}

// Appends the launch attributes: clusters of `cluster` CTAs along x (cluster > 1) and
// programmatic stream serialisation (pdl).  attr holds two entries.
inline void set_launch_attrs(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int cluster, bool pdl) {
    unsigned n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
}

template <int BN, int kMaj, bool kSplit, bool kSwiGLU, bool kSepC, int kKindT>
cudaError_t launch_gemm(const GemmParams& p, const GemmMaps& maps, int grid, cudaStream_t stream) {
    cudaError_t err = configure_gemm<BN, kMaj, kSplit, kSwiGLU, kSepC, kKindT>();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = TileCfg<BN, kSplit, kSwiGLU, kSepC>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    set_launch_attrs(cfg, attr, kSplit ? p.split : 1, p.pdl != 0);
    return cudaLaunchKernelEx(&cfg, fg_gemm_kernel<BN, kMaj, kSplit, kSwiGLU, kSepC, kKindT>, p, maps);
}

template <int BN, int kMaj, bool kSplit, bool kSwiGLU, bool kSepC, int kKindT>
cudaError_t max_active_clusters(int cluster, int* out) {
    cudaError_t err = configure_gemm<BN, kMaj, kSplit, kSwiGLU, kSepC, kKindT>();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = TileCfg<BN, kSplit, kSwiGLU, kSepC>::kSmemBytes;
    cudaLaunchAttribute attr[2];
    set_launch_attrs(cfg, attr, cluster, false);
    return cudaOccupancyMaxActiveClusters(out, fg_gemm_kernel<BN, kMaj, kSplit, kSwiGLU, kSepC, kKindT>, &cfg);
}

}  // namespace fg
