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
//
// A fourth kernel makes the weights of the FP8 x FP4 GEMMs ("FP4 with UE8M0 SF", the
// Chinese post's "Mega MoE" section): E2M1 codes with one UE8M0 scale per 32 K elements
// of a row (the MXFP4 block), the smallest power of two 2^e with amax <= 6 * 2^e.
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fg.h"
#include "fg_fp8.cuh"

namespace {

using fg::e4m3x4;
using fg::pow2_neg;
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
        const float sc = pow2_neg(e);
        uint32_t packed[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            packed[i] = e4m3x4(v[4 * i] * sc, v[4 * i + 1] * sc, v[4 * i + 2] * sc, v[4 * i + 3] * sc);
        *reinterpret_cast<uint4*>(q + (long long)row * K + k0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
    const uint32_t b1 = __shfl_sync(0xffffffffu, byte, 8);
    const uint32_t b2 = __shfl_sync(0xffffffffu, byte, 16);
    const uint32_t b3 = __shfl_sync(0xffffffffu, byte, 24);
    if (lane == 0) sf[(long long)w * sf_ld + row] = static_cast<int32_t>(byte | b1 << 8 | b2 << 16 | b3 << 24);
}

// MXFP4 scale exponent: the smallest e with amax <= 6 * 2^e.  With amax = fr * 2^ex,
// fr in [0.5, 1): amax / 2^(ex-3) = 8 fr lies in [4, 8), within 6 iff fr <= 0.75.
__device__ __forceinline__ int mxfp4_exponent(float amax) {
    if (!(amax > 0.0f)) return 0;
    int ex;
    const float fr = frexpf(amax, &ex);
    int e = fr <= 0.75f ? ex - 3 : ex - 2;
    return e < -127 ? -127 : (e > 126 ? 126 : e);   // a finite amax gives e <= 126 anyway
}

// One warp per (row, eight 128-wide K-groups): lane l holds K elements 4l..4l+3 of each of
// the warp's K-groups (eight independent 16-byte loads in flight per lane), eight lanes per
// 32-wide block.  The eight warps of a CTA take eight consecutive rows of the same K-groups,
// so their scale words are adjacent.  Codes: E2M1 round-to-nearest-even of x * 2^-e, the
// scaling an exact multiply by the power of two (e <= 126 for every finite amax, so 2^-e is
// a normal float), element 2i in bits 0-3 of byte i.  Measured on GB300 (32 x 4096 x 4096
// weights): one K-group per warp and ldexpf 821 us, four K-groups 486 us, eight 445 us, the
// multiply instead of ldexpf 420 us, both 396 us, paired conversions 377 us (0.95 of HBM).
__global__ void __launch_bounds__(256) quant_mxfp4_kernel(const float* __restrict__ w, long long rows, int N,
                                                          int K, uint8_t* __restrict__ q, int32_t* __restrict__ sf,
                                                          int sf_ld) {
    const int kgs = K / 128;
    const int kq = (kgs + 7) / 8;
    const int kg0 = static_cast<int>(blockIdx.x % kq) * 8;
    const long long row = (long long)(blockIdx.x / kq) * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const int nkg = kgs - kg0 < 8 ? kgs - kg0 : 8;
    float4 t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < nkg) t[i] = __ldg(reinterpret_cast<const float4*>(w + row * K + (kg0 + i) * 128) + lane);
    const long long g = row / N, n = row % N;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i >= nkg) break;   // warp-uniform
        float amax = fmaxf(fmaxf(fabsf(t[i].x), fabsf(t[i].y)), fmaxf(fabsf(t[i].z), fabsf(t[i].w)));
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int e = mxfp4_exponent(amax);
        const float sc = __int_as_float((127 - e) << 23);    // 2^-e
        const float v[4] = {t[i].x * sc, t[i].y * sc, t[i].z * sc, t[i].w * sc};
        // two codes per conversion, the pair's .x in the low nibble
        const uint32_t c01 = __nv_cvt_float2_to_fp4x2(make_float2(v[0], v[1]), __NV_E2M1, cudaRoundNearest);
        const uint32_t c23 = __nv_cvt_float2_to_fp4x2(make_float2(v[2], v[3]), __NV_E2M1, cudaRoundNearest);
        const uint32_t codes = (c01 & 0xFFu) | (c23 & 0xFFu) << 8;
        *reinterpret_cast<uint16_t*>(q + row * (K / 2) + (kg0 + i) * 64 + lane * 2) = static_cast<uint16_t>(codes);
        const uint32_t byte = static_cast<uint32_t>(e + 127);
        const uint32_t b1 = __shfl_sync(0xffffffffu, byte, 8);
        const uint32_t b2 = __shfl_sync(0xffffffffu, byte, 16);
        const uint32_t b3 = __shfl_sync(0xffffffffu, byte, 24);
        if (lane == 0) sf[(g * kgs + kg0 + i) * sf_ld + n] = static_cast<int32_t>(byte | b1 << 8 | b2 << 16 | b3 << 24);
    }
}

// The scale byte of K-group kg goes straight into its packed word (byte kg mod 4); the CTA
// of the last K-group also clears the word's bytes of K-groups past K, so every word ends
// up fully defined whatever the buffer held.
__device__ __forceinline__ void put_scale_byte(uint8_t* word, int kg, int num_kg, int e) {
    word[kg & 3] = static_cast<uint8_t>(e + 127);
    if (kg == num_kg - 1)
        for (int b = (kg & 3) + 1; b < 4; ++b) word[b] = 0;
}

// One CTA (8 warps, 16 rows each) per 128x128 block: (K-group, 128-row block, group).
__global__ void __launch_bounds__(256) quant_blocks_kernel(const float* __restrict__ w, int N, int K,
                                                           uint8_t* __restrict__ q, int32_t* __restrict__ sf,
                                                           int sf_ld, int kp) {
    __shared__ float red[8];
    const int kg = blockIdx.x, nb = blockIdx.y, g = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* base = w + (long long)g * N * K;
    uint8_t* qbase = q + (long long)g * N * K;
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
    const int e = scale_exponent(amax);
    const float sc = pow2_neg(e);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int row = nb * 128 + warp * 16 + r;
        if (row < N)
            *reinterpret_cast<uint32_t*>(qbase + (long long)row * K + kg * 128 + lane * 4) =
                e4m3x4(v[r][0] * sc, v[r][1] * sc, v[r][2] * sc, v[r][3] * sc);
    }
    if (threadIdx.x == 0)
        put_scale_byte(reinterpret_cast<uint8_t*>(sf + ((long long)g * kp + kg / 4) * sf_ld + nb), kg, K / 128, e);
}

// One CTA per (128-row K-group, 128 columns) of x[K][MN]: the tile is read from HBM once,
// straight into shared memory by 16-byte cp.async copies (all in flight together), each
// thread takes one column's amax there, and the codes leave as one 4-code word per row and
// four columns (coalesced).  64 KB per CTA: three CTAs share an SM, so one's copies overlap
// another's encoding.
constexpr int kColTile = 128;                     // columns per CTA
constexpr int kColSmem = 128 * kColTile * 4 + kColTile * 4;

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all_copies() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__global__ void __launch_bounds__(256) quant_cols_kernel(const float* __restrict__ x, int K, int MN,
                                                         uint8_t* __restrict__ q, int32_t* __restrict__ sf,
                                                         int sf_ld) {
    extern __shared__ __align__(16) float tile[];  // [128][kColTile], then the exponents
    int* ex = reinterpret_cast<int*>(tile + 128 * kColTile);
    const int kg = blockIdx.x;
    const int c0 = blockIdx.y * kColTile;
    const int ncols = min(kColTile, MN - c0);      // a multiple of 16
    const int t = threadIdx.x;
    const float* src = x + (long long)kg * 128 * MN + c0;
    // stage: 128 rows x ncols/4 float4 groups; thread t copies group t % 32 of rows t / 32 + 8i
    const int g4 = t & 31, r0 = t >> 5;
    const uint32_t tile_u32 = static_cast<uint32_t>(__cvta_generic_to_shared(tile));
    if (4 * g4 < ncols) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = r0 + 8 * i;
            cp_async_16(tile_u32 + static_cast<uint32_t>((r * kColTile + 4 * g4) * 4), src + (long long)r * MN + 4 * g4);
        }
    }
    cp_async_wait_all_copies();
    __syncthreads();
    if (t < ncols) {
        float amax = 0.0f;
#pragma unroll 8
        for (int r = 0; r < 128; ++r) amax = fmaxf(amax, fabsf(tile[r * kColTile + t]));
        const int e = scale_exponent(amax);
        ex[t] = e;
        put_scale_byte(reinterpret_cast<uint8_t*>(sf + (long long)(kg / 4) * sf_ld + c0 + t), kg, K / 128, e);
    }
    __syncthreads();
    uint8_t* dst = q + (long long)kg * 128 * MN + c0;
    if (4 * g4 < ncols) {
        const float s0 = pow2_neg(ex[4 * g4]), s1 = pow2_neg(ex[4 * g4 + 1]);
        const float s2 = pow2_neg(ex[4 * g4 + 2]), s3 = pow2_neg(ex[4 * g4 + 3]);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = r0 + 8 * i;
            const float4 v = reinterpret_cast<const float4*>(tile + r * kColTile)[g4];
            *reinterpret_cast<uint32_t*>(dst + (long long)r * MN + 4 * g4) = e4m3x4(v.x * s0, v.y * s1, v.z * s2, v.w * s3);
        }
    }
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
    quant_blocks_kernel<<<dim3(K / 128, nblk, G), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        w, N, K, q, sf, align4(nblk), kp);
    return finish_launch();
}

int fg_quantize_mxfp4(int G, int N, int K, const float* w, uint8_t* q, int32_t* sf, fg_stream_t stream) {
    if (G < 1 || N < 1 || K < 128 || K % 128 != 0 || !w || !q || !sf || !al16(w) || !al16(q) || !al16(sf))
        return FG_ERR_INVALID_ARG;
    int dev;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return FG_ERR_CUDA; }
    const long long rows = (long long)G * N;
    const long long blocks = (rows + 7) / 8 * ((K / 128 + 7) / 8);
    if (blocks > 0x7fffffffLL) return FG_ERR_INVALID_ARG;
    quant_mxfp4_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        w, rows, N, K, q, sf, align4(N));
    return finish_launch();
}

int fg_quantize_1x128_cols(int K, int MN, const float* x, uint8_t* q, int32_t* sf, fg_stream_t stream) {
    if (K < 0 || K % 128 != 0 || MN < 1 || MN % 16 != 0 || !x || !q || !sf || !al16(x) || !al16(q) ||
        !al16(sf))
        return FG_ERR_INVALID_ARG;
    if (K == 0) return FG_OK;
    int dev;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return FG_ERR_CUDA; }
    const int cblk = (MN + kColTile - 1) / kColTile;
    if (cblk > 65535) return FG_ERR_INVALID_ARG;
    if (dev < 0 || dev >= 256) return FG_ERR_CUDA;
    {   // the staged tile's shared memory, allowed once per device
        static std::mutex mu;
        static bool configured[256] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (!configured[dev]) {
            if (cudaFuncSetAttribute(quant_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kColSmem) !=
                cudaSuccess) {
                cudaGetLastError();
                return FG_ERR_CUDA;
            }
            configured[dev] = true;
        }
    }
    quant_cols_kernel<<<dim3(K / 128, cblk), 256, kColSmem, reinterpret_cast<cudaStream_t>(stream)>>>(
        x, K, MN, q, sf, align4(MN));
    return finish_launch();
}

}  // extern "C"
