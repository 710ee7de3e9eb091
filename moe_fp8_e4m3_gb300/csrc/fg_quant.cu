// fg_quant.cu - FP32 -> E4M3 quantisation with UE8M0 power-of-two scales, written
// straight into the packed, MN-major, TMA-aligned scale layout the GEMMs read.
//
// The pages leave the FP8 cast to the user and list the layout helpers the library
// offers for it ("DeepGEMM Documentation", section 4 note on FP8 casting, and section 10
// "Use DeepGEMM Utility Functions": transform_sf_into_required_layout,
// get_mn_major_tma_aligned_packed_ue8m0_tensor,
// get_k_grouped_mn_major_tma_aligned_packed_ue8m0_tensor).  Three granularities:
//   rows    1x128 groups along the contiguous K axis of x[rows][K]      (activations)
//   blocks  128x128 blocks of w[G][N][K]                                (weights)
//   cols    1x128 groups along the leading axis of x[K][MN]             (K-grouped operands)
// Scale of a group: the smallest power of two 2^e with amax <= 448 * 2^e (byte e+127,
// clamped to [0, 254]; an all-zero group gets byte 127).  Code: E4M3
// round-to-nearest-even of x * 2^-e, which is exact scaling and never exceeds 448.
// All three kernels are HBM-bound streaming passes: one read of x, one write of q.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fg.h"
#include "fg_fp8.cuh"

namespace {

using fg::e4m3;
using fg::scale_exponent;

// One warp per (row, packed word): 512 consecutive K elements, 16 per lane, 8 lanes per
// 128-group.
__global__ void __launch_bounds__(256) quant_rows_kernel(const float* __restrict__ x, int rows, int K,
                                                         uint8_t* __restrict__ q, int32_t* __restrict__ sf,
                                                         int sf_ld, long long num_items) {
    const long long item = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (item >= num_items) return;
    const int lane = threadIdx.x & 31;
    const int kp = (K + 511) / 512;
    const int row = static_cast<int>(item / kp), w = static_cast<int>(item % kp);
    const int k0 = w * 512 + lane * 16;
    const bool active = k0 < K;
    float v[16];
    float amax = 0.0f;
    if (active) {
        const float4* src = reinterpret_cast<const float4*>(x + (long long)row * K + k0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 t = __ldg(src + i);
            v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = scale_exponent(amax);
    const uint32_t byte = active ? static_cast<uint32_t>(e + 127) : 0u;
    if (active) {
        uint32_t packed[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) word |= e4m3(ldexpf(v[4 * i + j], -e)) << (8 * j);
            packed[i] = word;
        }
        *reinterpret_cast<uint4*>(q + (long long)row * K + k0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
    const uint32_t b1 = __shfl_sync(0xffffffffu, byte, 8);
    const uint32_t b2 = __shfl_sync(0xffffffffu, byte, 16);
    const uint32_t b3 = __shfl_sync(0xffffffffu, byte, 24);
    if (lane == 0) sf[(long long)w * sf_ld + row] = static_cast<int32_t>(byte | b1 << 8 | b2 << 16 | b3 << 24);
}

// One CTA (8 warps) per (group, 128-row block, packed word): up to four 128x128 blocks.
__global__ void __launch_bounds__(256) quant_blocks_kernel(const float* __restrict__ w, int N, int K,
                                                           uint8_t* __restrict__ q, int32_t* __restrict__ sf,
                                                           int sf_ld, int kp, int nblk) {
    __shared__ float red[8];
    const int g = blockIdx.z, nb = blockIdx.y, wd = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* base = w + (long long)g * N * K;
    uint8_t* qbase = q + (long long)g * N * K;
    uint32_t word = 0;
    for (int j = 0; j < 4; ++j) {
        const int kg = wd * 4 + j;
        if (kg * 128 >= K) break;
        float v[16][4];
        float amax = 0.0f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int row = nb * 128 + warp * 16 + r;
            if (row < N) {
                const float4 t = __ldg(reinterpret_cast<const float4*>(base + (long long)row * K + kg * 128) + lane);
                v[r][0] = t.x; v[r][1] = t.y; v[r][2] = t.z; v[r][3] = t.w;
            } else {
                v[r][0] = v[r][1] = v[r][2] = v[r][3] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(v[r][i]));
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
        __syncthreads();
        const int e = scale_exponent(amax);
        word |= static_cast<uint32_t>(e + 127) << (8 * j);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int row = nb * 128 + warp * 16 + r;
            if (row < N) {
                uint32_t b = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) b |= e4m3(ldexpf(v[r][i], -e)) << (8 * i);
                *reinterpret_cast<uint32_t*>(qbase + (long long)row * K + kg * 128 + lane * 4) = b;
            }
        }
    }
    if (threadIdx.x == 0) sf[((long long)g * kp + wd) * sf_ld + nb] = static_cast<int32_t>(word);
    (void)nblk;
}

// One thread per column of x[K][MN]; a CTA covers 256 columns of one packed word (512
// rows).  Two passes per 128-row group: amax, then encode (the second read hits L2).
__global__ void __launch_bounds__(256) quant_cols_kernel(const float* __restrict__ x, int K, int MN,
                                                         uint8_t* __restrict__ q, int32_t* __restrict__ sf,
                                                         int sf_ld) {
    const int col = blockIdx.x * 256 + threadIdx.x;
    const int wd = blockIdx.y;
    if (col >= MN) return;
    uint32_t word = 0;
    for (int j = 0; j < 4; ++j) {
        const int kg = wd * 4 + j;
        if (kg * 128 >= K) break;
        const float* src = x + (long long)kg * 128 * MN + col;
        float amax = 0.0f;
#pragma unroll 8
        for (int r = 0; r < 128; ++r) amax = fmaxf(amax, fabsf(__ldg(src + (long long)r * MN)));
        const int e = scale_exponent(amax);
        word |= static_cast<uint32_t>(e + 127) << (8 * j);
        uint8_t* dst = q + (long long)kg * 128 * MN + col;
#pragma unroll 8
        for (int r = 0; r < 128; ++r)
            dst[(long long)r * MN] = static_cast<uint8_t>(e4m3(ldexpf(__ldg(src + (long long)r * MN), -e)));
    }
    sf[(long long)wd * sf_ld + col] = static_cast<int32_t>(word);
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int align4(int x) { return (x + 3) / 4 * 4; }

int finish_launch() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FG_OK : FG_ERR_CUDA;
}

}  // namespace

extern "C" {

int fg_quantize_1x128_rows(int rows, int K, const float* x, uint8_t* q, int32_t* sf, fg_stream_t stream) {
    if (rows < 0 || K < 128 || K % 128 != 0 || !x || !q || !sf || !al16(x) || !al16(q) || !al16(sf))
        return FG_ERR_INVALID_ARG;
    if (rows == 0) return FG_OK;
    int dev;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return FG_ERR_CUDA; }
    const long long items = (long long)rows * ((K + 511) / 512);
    const long long blocks = (items + 7) / 8;
    if (blocks > 0x7fffffffLL) return FG_ERR_INVALID_ARG;
    quant_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        x, rows, K, q, sf, align4(rows), items);
    return finish_launch();
}

int fg_quantize_128x128_blocks(int G, int N, int K, const float* w, uint8_t* q, int32_t* sf,
                               fg_stream_t stream) {
    if (G < 1 || G > 65535 || N < 1 || K < 128 || K % 128 != 0 || !w || !q || !sf || !al16(w) || !al16(q) ||
        !al16(sf))
        return FG_ERR_INVALID_ARG;
    int dev;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return FG_ERR_CUDA; }
    const int kp = (K + 511) / 512, nblk = (N + 127) / 128;
    if (nblk > 65535) return FG_ERR_INVALID_ARG;
    quant_blocks_kernel<<<dim3(kp, nblk, G), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        w, N, K, q, sf, align4(nblk), kp, nblk);
    return finish_launch();
}

int fg_quantize_1x128_cols(int K, int MN, const float* x, uint8_t* q, int32_t* sf, fg_stream_t stream) {
    if (K < 0 || K % 128 != 0 || MN < 1 || MN % 16 != 0 || !x || !q || !sf || !al16(x) || !al16(q) ||
        !al16(sf))
        return FG_ERR_INVALID_ARG;
    if (K == 0) return FG_OK;
    int dev;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return FG_ERR_CUDA; }
    const int kp = (K + 511) / 512;
    if (kp > 65535) return FG_ERR_INVALID_ARG;
    quant_cols_kernel<<<dim3((MN + 255) / 256, kp), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        x, K, MN, q, sf, align4(MN));
    return finish_launch();
}

}  // extern "C"
