// fg_api.cu - the C ABI declared in include/fg.h: host-side validation, TMA tensor-map
// encoding, tile-size choice and launch of the persistent FP8 GEMM kernels.
//
// No allocation happens per call.  Per device the library keeps the SM count and the
// device address of its status word; the TMA encoder is fetched once from the driver.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fg.h"
#include "fg_launch.h"
#include "fg_mqa.cuh"

// Device status word: first contract violation or wait time-out since the last read.
__device__ int g_fg_status = 0;
// The value taken out of the status word by fg_get_device_error (read back to the host).
__device__ int g_fg_status_taken = 0;

namespace {
// Reads and clears the status word in one atomic exchange, in stream order: an event a
// kernel on another stream records at the same moment lands either in this read or in
// the word for the next one, never nowhere.
__global__ void take_status_kernel(int* status, int* taken) { *taken = atomicExch(status, 0); }
}  // namespace

namespace {

using fg::GemmParams;

constexpr int kMaxDevices = 256;
constexpr unsigned long long kDefaultTimeoutNs = 4000000000ull;  // 4 s per wait

constexpr int kBnChoices[5] = {64, 128, 192, 224, 256};

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int* status = nullptr;
    int* taken = nullptr;
    // resident split-K clusters of the dense NT kernel per tile width and cluster size
    // 2/4/8; 0 = not queried yet, -1 = query failed
    int clusters[5][3] = {};
};

std::mutex g_mu;
std::mutex g_take_mu;   // one status read at a time (they share the device's take slot)
DeviceState g_dev[kMaxDevices];
int g_num_sms_limit = 0;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;
int g_debug_stall = 0;
int g_pdl = 1;
unsigned long long g_timeout_ns = kDefaultTimeoutNs;

int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return FG_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return FG_ERR_CUDA;
        }
        void* ptr = nullptr;
        void* ptr_taken = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_fg_status) != cudaSuccess ||
            cudaGetSymbolAddress(&ptr_taken, g_fg_status_taken) != cudaSuccess) {
            cudaGetLastError();
            return FG_ERR_CUDA;
        }
        st.num_sms = sms;
        st.status = static_cast<int*>(ptr);
        st.taken = static_cast<int*>(ptr_taken);
        st.ready = true;
    }
    if (!g_encode_tried) {
        g_encode_tried = true;
        cudaDriverEntryPointQueryResult q{};
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    }
    if (!g_encode) return FG_ERR_CUDA;
    *out = &st;
    return FG_OK;
}

int sms_in_use(const DeviceState& st) {
    return (g_num_sms_limit > 0 && g_num_sms_limit < st.num_sms) ? g_num_sms_limit : st.num_sms;
}

// Split-K clusters of `cluster` CTAs (2, 4 or 8) that fit on the device at once.
int resident_clusters(DeviceState& st, int bn, int cluster) {
    int bi = 0;
    while (bi < 4 && kBnChoices[bi] != bn) ++bi;
    const int ci = cluster == 2 ? 0 : (cluster == 4 ? 1 : 2);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (st.clusters[bi][ci] != 0) return st.clusters[bi][ci] > 0 ? st.clusters[bi][ci] : 0;
    }
    int n = 0;
    cudaError_t e = cudaErrorInvalidValue;
    switch (bn) {
        case 64: e = fg::max_active_clusters<64, fg::kMajNT, true, false, false, fg::kDense>(cluster, &n); break;
        case 128: e = fg::max_active_clusters<128, fg::kMajNT, true, false, false, fg::kDense>(cluster, &n); break;
        case 192: e = fg::max_active_clusters<192, fg::kMajNT, true, false, false, fg::kDense>(cluster, &n); break;
        case 224: e = fg::max_active_clusters<224, fg::kMajNT, true, false, false, fg::kDense>(cluster, &n); break;
        default: e = fg::max_active_clusters<256, fg::kMajNT, true, false, false, fg::kDense>(cluster, &n); break;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        n = -1;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    st.clusters[bi][ci] = n;
    return n > 0 ? n : 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
int align4(int x) { return (x + 3) / 4 * 4; }
int ceil_div(int a, int b) { return (a + b - 1) / b; }

// 2-D tiled tensor map over a row-major [outer][inner] array with the given row pitch.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
               uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box,
                                elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D tiled tensor map over [outer2][outer1][inner] (pitches in bytes).
bool encode_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
               uint64_t outer1, uint64_t outer2, uint64_t pitch1, uint64_t pitch2, uint32_t box_inner,
               uint32_t box_outer1, CUtensorMapSwizzle swizzle) {
    cuuint64_t dims[3] = {inner, outer1, outer2};
    cuuint64_t strides[2] = {pitch1, pitch2};
    cuuint32_t box[3] = {box_inner, box_outer1, 1};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    const CUresult r = g_encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box,
                                elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// C/D maps of a [rows][N] output: boxes of box_rows rows x 128 bytes (32 FP32 or 64 BF16
// columns), 128-byte swizzle, matching the epilogue's shared-memory slots (128 rows for a
// whole block, 32 rows for one epilogue warp's rows).
bool encode_out_2d(CUtensorMap* map, const void* base, int n, long long rows, bool f32, uint32_t box_rows) {
    const uint32_t esz = f32 ? 4 : 2;
    return encode_2d(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base,
                     (uint64_t)n, (uint64_t)rows, (uint64_t)n * esz, 128 / esz, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// D map of a [rows][N] output: one epilogue warp's 32 rows per box.
bool encode_d_maps(fg::GemmMaps& gm, const void* d, int n, long long rows, bool f32) {
    return encode_out_2d(&gm.d, d, n, rows, f32, 32);
}

// C map of a [rows][N] FP32 input: one epilogue warp's 32 rows per box.
bool encode_c_maps(fg::GemmMaps& gm, const float* c, int n, long long rows) {
    return encode_out_2d(&gm.c, c, n, rows, true, 32);
}

bool print_configs() {
    const char* e = std::getenv("FG_PRINT_CONFIGS");
    return e && e[0] == '1';
}

// Optional override of the N tile (tuning aid): FG_FORCE_BN=64|128|192|224|256.
int forced_bn() {
    const char* e = std::getenv("FG_FORCE_BN");
    return e ? std::atoi(e) : 0;
}

// Optional override of the dense split-K cluster size (tuning aid): FG_FORCE_SPLIT=1|2|4|8.
// A forced split that cannot run (too many tiles for one resident wave of clusters)
// falls back to the model's choice.
int forced_split() {
    const char* e = std::getenv("FG_FORCE_SPLIT");
    return e ? std::atoi(e) : 0;
}

// N-tile choice.  Cost model: the busiest SM runs ceil(tiles / SMs) tiles, each costing
// about (BN + 32) column units (the 32 stands for the A re-read and fixed per-tile work).
// BN=256 has a single TMEM accumulator, so its epilogue does not overlap the next tile's
// MMAs: it is charged 15 % more, and with a heavy epilogue (a C, or an FP32 D: 4 bytes per
// output) it is not considered.  Measured on GB300: 4096 x 7168 x 2048 FP32 D without C,
// BN=224 67 us against BN=256 74 us; BF16 D, masked 32 x 256 x 4096 x 2048 62.1 us against
// 63.9 us and contiguous 32 x 4096 x 4096 137.9 us against 140.2 us.  Where two widths cost
// the same, the one whose last wave leaves fewer SMs idle is taken (then the order of the
// list): the same GEMM with an FP32 C, 7 waves of 224 (the last one 112 tiles) or exactly 8
// of 192, ran 70.8 us at BN=224 and 69.7 us at 192 as the first GEMM of the dense pair (step
// 1467 against 1485 TFLOP/s over ten runs each; 73.7 against 74.0 us alone).
// The FP8 x FP4 variants exist at two widths, 128 and 224 (fp4 restricts the choice to them).
bool fp4_width(int bn) { return bn == 128 || bn == 224; }

int choose_bn_nt(long long row_blocks, int n, int sms, bool heavy_epilogue, bool fp4 = false) {
    const int f = forced_bn();
    if ((f == 64 || f == 128 || f == 192 || f == 224 || f == 256) && (!fp4 || fp4_width(f))) return f;
    int best = 128;
    double best_cost = -1.0;
    long long best_idle = 0;
    for (int bn : {224, 256, 192, 128, 64}) {
        if (heavy_epilogue && bn == 256) continue;
        if (fp4 && !fp4_width(bn)) continue;
        const long long tiles = row_blocks * ceil_div(n, bn);
        const long long waves = (tiles + sms - 1) / sms;
        const long long idle = waves * sms - tiles;     // SMs without a tile in the last wave
        const double cost = static_cast<double>(waves * (bn + 32)) * (bn == 256 ? 1.15 : 1.0);
        if (best_cost < 0 || cost < best_cost || (cost == best_cost && idle < best_idle)) {
            best = bn;
            best_cost = cost;
            best_idle = idle;
        }
    }
    return best;
}

// Dense NT tiling: N tile and split-K cluster size.  Without a split the N tile is
// choose_bn_nt's.  A split-K cluster of s CTAs needs every tile's cluster resident in one
// wave; the choice between the two compares estimated times (microseconds):
//     waves * ceil(nkb / s) * t_kb(BN) + t_x(s)
// t_kb is the steady-state time of one K-group per CTA and t_x(s) the partial-tile
// exchange plus cluster barriers, both measured on a 64 x 7168 x 4096 GEMM on GB300 with
// all SMs busy and L2 flushed (TMA latency bound: deeper rings of narrow tiles keep up).
double t_kb_us(int bn) {
    switch (bn) {
        case 64: return 0.36;
        case 128: return 0.37;
        case 192: return 0.50;
        default: return 0.61;
    }
}
// t_x: the split-K epilogue (partials through distributed shared memory, cluster barriers)
// over a plain one; per-CTA timelines on GB300 put the 2-CTA exchange at ~3.6 us against
// ~1 us (and 128x256x512 runs in 8.6 us unsplit against 11.6 us in 2-CTA clusters).
double t_x_us(int s) { return s <= 1 ? 0.0 : (s == 2 ? 2.5 : (s == 4 ? 4.0 : 6.0)); }

struct DenseTiling {
    int bn;
    int split;
};
// fp4: the FP8 x FP4 variants (unsplit at 128 and 224, split-K clusters at 128).
DenseTiling choose_dense_tiling(DeviceState& st, int num_mb, int n, int k, int sms, bool heavy_epilogue,
                                bool fp4 = false) {
    const int fb = forced_bn(), fs = forced_split();
    const int nkb = k / 128;
    DenseTiling best{choose_bn_nt(num_mb, n, sms, heavy_epilogue, fp4), 1};
    const long long tiles1 = (long long)num_mb * ceil_div(n, best.bn);
    double best_t = (double)((tiles1 + sms - 1) / sms) * nkb * t_kb_us(best.bn);
    if (fs == 1) return best;
    for (int bn : {256, 224, 192, 128, 64}) {
        if (fb && bn != fb) continue;
        if (fp4 && bn != 128) continue;
        const long long tiles = (long long)num_mb * ceil_div(n, bn);
        for (int s : {2, 4, 8}) {
            if (fs && s != fs) continue;
            if (tiles * s > sms) continue;
            if (!fs && nkb < 2 * s) continue;
            if (tiles > resident_clusters(st, bn, s)) continue;
            const double t = ceil_div(nkb, s) * t_kb_us(bn) + t_x_us(s);
            if (fs || t < best_t) {
                best = DenseTiling{bn, s};
                best_t = t;
                if (fs) return best;
            }
        }
    }
    return best;
}

int choose_bn_tn(long long row_blocks, int n, int sms, bool heavy_epilogue) {
    const int f = forced_bn();
    if (f == 128 || f == 256) return f;
    if (heavy_epilogue) return 128;
    return row_blocks * ceil_div(n, 256) >= sms ? 256 : 128;
}

// L2 prefetch of a single-tile CTA's B before its grid-dependency wait (FG_PREFETCH_B=0 disables it).
int prefetch_b_enabled() {
    const char* e = std::getenv("FG_PREFETCH_B");
    return e && e[0] == '0' ? 0 : 1;
}

void fill_common(GemmParams& p, const DeviceState& st) {
    p.split = 1;
    p.a_box_rows = 128;
    p.status = st.status;
    p.timeout_ns = g_timeout_ns;
    p.debug_stall = g_debug_stall;
    p.pdl = g_pdl;
}

// C is an array of its own (not D): launch the variant that prefetches it into slots.
bool separate_c(const GemmParams& p) { return p.has_c && !p.c_in_d; }

// One NT launch of the variant family <kSplit, kSepC, kKind> at tile width bn (BN=256 has no
// C slots: its separate-C calls take the plain variant, C landing in the store slot).
template <bool kSplit, bool kSepC, int kKind>
cudaError_t launch_nt_bn(int bn, const GemmParams& p, const fg::GemmMaps& gm, int grid, cudaStream_t s) {
    switch (bn) {
        case 64: return fg::launch_gemm<64, fg::kMajNT, kSplit, false, kSepC, kKind>(p, gm, grid, s);
        case 128: return fg::launch_gemm<128, fg::kMajNT, kSplit, false, kSepC, kKind>(p, gm, grid, s);
        case 192: return fg::launch_gemm<192, fg::kMajNT, kSplit, false, kSepC, kKind>(p, gm, grid, s);
        case 224: return fg::launch_gemm<224, fg::kMajNT, kSplit, false, kSepC, kKind>(p, gm, grid, s);
        default: return fg::launch_gemm<256, fg::kMajNT, kSplit, false, false, kKind>(p, gm, grid, s);
    }
}

// One FP8 x FP4 launch (B packed E2M1): tile width 128 or 224, split-K clusters at 128.
template <bool kSplit, bool kSepC, int kKind>
cudaError_t launch_fp4_bn(int bn, const GemmParams& p, const fg::GemmMaps& gm, int grid, cudaStream_t s) {
    if (bn == 128) return fg::launch_gemm<128, fg::kMajNTF4, kSplit, false, kSepC, kKind>(p, gm, grid, s);
    if constexpr (!kSplit) {
        if (bn == 224) return fg::launch_gemm<224, fg::kMajNTF4, false, false, kSepC, kKind>(p, gm, grid, s);
    }
    return cudaErrorInvalidValue;
}

int launch_fp4(int bn, const GemmParams& p, const fg::GemmMaps& gm, int grid, cudaStream_t s) {
    cudaError_t e;
    if (p.split > 1) e = launch_fp4_bn<true, false, fg::kDense>(bn, p, gm, grid, s);
    else if (p.kind == fg::kContiguous) e = launch_fp4_bn<false, false, fg::kContiguous>(bn, p, gm, grid, s);
    else if (p.kind == fg::kMasked) e = launch_fp4_bn<false, false, fg::kMasked>(bn, p, gm, grid, s);
    else if (separate_c(p)) e = launch_fp4_bn<false, true, fg::kDense>(bn, p, gm, grid, s);
    else e = launch_fp4_bn<false, false, fg::kDense>(bn, p, gm, grid, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FG_ERR_CUDA;
    }
    return FG_OK;
}

int launch_nt(int bn, const GemmParams& p, const fg::GemmMaps& gm, int grid, cudaStream_t s) {
    cudaError_t e;
    if (p.split > 1) e = launch_nt_bn<true, false, fg::kDense>(bn, p, gm, grid, s);
    else if (p.kind == fg::kContiguous) e = launch_nt_bn<false, false, fg::kContiguous>(bn, p, gm, grid, s);
    else if (p.kind == fg::kMasked) e = launch_nt_bn<false, false, fg::kMasked>(bn, p, gm, grid, s);
    else if (separate_c(p)) e = launch_nt_bn<false, true, fg::kDense>(bn, p, gm, grid, s);
    else e = launch_nt_bn<false, false, fg::kDense>(bn, p, gm, grid, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FG_ERR_CUDA;
    }
    return FG_OK;
}

// Gate-up weights b [G][2I][K] seen as [2G halves][I rows][K]: a {128 K, 128 rows, 2 halves}
// box brings a tile's gate rows and the matching up rows in one copy.  fp4: b [G][2I][K/2]
// packed E2M1, unpacked by the tensor map as for encode_b_nt.
bool encode_swiglu_b(CUtensorMap* map, const void* b, int K, int I, int G, bool fp4) {
    const cuuint64_t row_bytes = fp4 ? (cuuint64_t)K / 2 : (cuuint64_t)K;
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)I, (cuuint64_t)2 * G};
    cuuint64_t strides[2] = {row_bytes, (cuuint64_t)I * row_bytes};
    cuuint32_t box[3] = {128, 128, 2};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    return g_encode(map, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                    const_cast<void*>(b), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_swiglu(bool fp4, const GemmParams& p, const fg::GemmMaps& gm, int grid, cudaStream_t s) {
    const bool masked = p.kind == fg::kMasked;
    const cudaError_t e =
        fp4 ? (masked ? fg::launch_gemm<256, fg::kMajNTF4, false, true, false, fg::kMasked>(p, gm, grid, s)
                      : fg::launch_gemm<256, fg::kMajNTF4, false, true, false, fg::kContiguous>(p, gm, grid, s))
            : (masked ? fg::launch_gemm<256, fg::kMajNT, false, true, false, fg::kMasked>(p, gm, grid, s)
                      : fg::launch_gemm<256, fg::kMajNT, false, true, false, fg::kContiguous>(p, gm, grid, s));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FG_ERR_CUDA;
    }
    return FG_OK;
}

// One launch with an MN-major operand at tile width bn (128 or 256; 224 as well for TT) of
// layout kKind; a separate C takes the variant with C slots where the width has them (128,
// and 224 for TT).
template <int kMaj, int kKind>
cudaError_t launch_mn_bn(int bn, bool sep, const GemmParams& p, const fg::GemmMaps& gm, int grid, cudaStream_t s) {
    if (bn == 128) {
        if (sep) return fg::launch_gemm<128, kMaj, false, false, true, kKind>(p, gm, grid, s);
        return fg::launch_gemm<128, kMaj, false, false, false, kKind>(p, gm, grid, s);
    }
    if constexpr (kMaj == fg::kMajTT) {
        if (bn == 224) {
            if (sep) return fg::launch_gemm<224, kMaj, false, false, true, kKind>(p, gm, grid, s);
            return fg::launch_gemm<224, kMaj, false, false, false, kKind>(p, gm, grid, s);
        }
    }
    return fg::launch_gemm<256, kMaj, false, false, false, kKind>(p, gm, grid, s);
}

// Variants with an MN-major operand: dense TN / NN / TT, the K-grouped TN GEMM and the
// M-grouped contiguous NN GEMM (the grouped layouts take no separate C except K-grouped).
int launch_mn(int maj, int bn, const GemmParams& p, const fg::GemmMaps& gm, int grid, cudaStream_t s) {
    cudaError_t e;
    const bool sep = separate_c(p);
    const bool dense = p.kind == fg::kDense;
    if (maj == fg::kMajTN)
        e = dense ? launch_mn_bn<fg::kMajTN, fg::kDense>(bn, sep, p, gm, grid, s)
                  : launch_mn_bn<fg::kMajTN, fg::kKGrouped>(bn, sep, p, gm, grid, s);
    else if (maj == fg::kMajNN)
        e = dense ? launch_mn_bn<fg::kMajNN, fg::kDense>(bn, sep, p, gm, grid, s)
                  : launch_mn_bn<fg::kMajNN, fg::kContiguous>(bn, false, p, gm, grid, s);
    else
        e = launch_mn_bn<fg::kMajTT, fg::kDense>(bn, sep, p, gm, grid, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FG_ERR_CUDA;
    }
    return FG_OK;
}

// Shared checks of the NT operands: FP8 A/B and the packed scale arrays.  Packed FP4 B
// (fp4) must start on a 32-byte boundary (the unpacking TMA form's rule).
int check_nt_operands(int n, int k, const void* a, const void* sfa, const void* b,
                      const void* sfb, const void* d, int d_dtype, bool fp4 = false) {
    if (n < 16 || n % 16 != 0 || k < 128 || k % 128 != 0) return FG_ERR_INVALID_ARG;
    if (d_dtype != FG_BF16 && d_dtype != FG_F32) return FG_ERR_INVALID_ARG;
    if (!a || !sfa || !b || !sfb || !d) return FG_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d))
        return FG_ERR_INVALID_ARG;
    if (fp4 && (reinterpret_cast<uintptr_t>(b) & 31u) != 0) return FG_ERR_INVALID_ARG;
    return FG_OK;
}

// B tensor map of an NT call over `rows` rows of K: E4M3 bytes, or packed E2M1 codes (fp4)
// unpacked by the TMA unit into 16-byte chunks of 16 codes (8 bytes of codes, 8 of padding),
// the shared-memory form of a sub-byte tcgen05 operand, so a 128-code box row takes 128 bytes.
bool encode_b_nt(CUtensorMap* map, const void* b, int K, uint64_t rows, int bn, bool fp4) {
    if (fp4)
        return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, b, K, rows, (uint64_t)K / 2, 128, bn,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, K, rows, K, 128, bn, CU_TENSOR_MAP_SWIZZLE_128B);
}

// B scales: one per 128x128 block, packed per four K-groups; FP4 B: one per row and 32-wide
// block, one word (four blocks) per row and K-group.
void set_b_scales(GemmParams& p, int N, int K, bool fp4) {
    p.sfb_ld = fp4 ? align4(N) : align4(ceil_div(N, 128));
    p.sfb_per_row = fp4 ? 1 : 0;
    p.sfb_gstride = (long long)(fp4 ? K / 128 : ceil_div(K, 512)) * p.sfb_ld;
}

// Dense NT GEMM; fp4: B packed E2M1 with 1x32 scales (the FP8 x FP4 GEMM).
int dense_nt(bool fp4, int M, int N, int K, const uint8_t* a, const int32_t* sfa, const uint8_t* b,
             const int32_t* sfb, const float* c, void* d, int d_dtype, fg_stream_t stream) {
    if (M < 0) return FG_ERR_INVALID_ARG;
    int rc = check_nt_operands(N, K, a, sfa, b, sfb, d, d_dtype, fp4);
    if (rc) return rc;
    if (c && !aligned16(c)) return FG_ERR_INVALID_ARG;
    if (c && d_dtype != FG_F32) return FG_ERR_UNSUPPORTED;
    if (M == 0) return FG_OK;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st))) return rc;
    const int sms = sms_in_use(*st);
    const int num_mb = ceil_div(M, 128);
    const DenseTiling tiling = choose_dense_tiling(*st, num_mb, N, K, sms, c != nullptr || d_dtype == FG_F32, fp4);
    const int bn = tiling.bn;
    GemmParams p{};
    fill_common(p, *st);
    p.kind = fg::kDense;
    p.M = M; p.N = N; p.K = K; p.G = 1;
    p.d_f32 = d_dtype == FG_F32; p.has_c = c != nullptr;
    p.c_in_d = c != nullptr && static_cast<const void*>(c) == d;
    p.num_mb = num_mb;
    p.num_nb = ceil_div(N, bn);
    p.sfa = sfa; p.sfb = sfb;
    p.sfa_ld = align4(M);
    set_b_scales(p, N, K, fp4);
    p.sfa_rows = M;
    p.d = d;
    p.c = c;
    p.split = tiling.split;
    // a single row block of at most 64 rows: load only those rows of A (the MMA still
    // reads 128 rows of shared memory; rows past M produce accumulator rows never stored)
    p.a_box_rows = M <= 64 ? 64 : 128;
    fg::GemmMaps gm;
    std::memset(&gm, 0, sizeof(gm));
    CUtensorMap &ma = gm.a, &mb = gm.b, &mc = gm.c;
    std::memset(&mc, 0, sizeof(mc));
    if (!encode_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, M, K, 128, p.a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_b_nt(&mb, b, K, N, bn, fp4) ||
        !encode_d_maps(gm, d, N, M, p.d_f32) || (c && !encode_c_maps(gm, c, N, M)))
        return FG_ERR_INVALID_ARG;
    const long long tiles = (long long)p.num_mb * p.num_nb;
    // split-K: one tile per cluster, all clusters resident
    const int grid = p.split > 1 ? (int)tiles * p.split : (int)(tiles < sms ? tiles : sms);
    // one tile per CTA (or cluster): its B can be prefetched into L2 before the dependency wait
    p.prefetch_b = g_pdl && (p.split > 1 || tiles <= sms) && prefetch_b_enabled();
    if (print_configs())
        std::fprintf(stderr, "[fg] %s M=%d N=%d K=%d BN=%d split=%d tiles=%lld grid=%d\n",
                     fp4 ? "fp8_fp4_gemm_nt" : "fp8_gemm_nt", M, N, K, bn, p.split, tiles, grid);
    if (fp4) return launch_fp4(bn, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
    return launch_nt(bn, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
}

// M-grouped contiguous GEMM; b_nmajor: B stored [G][K][N] (NN) instead of [G][N][K] (NT);
// fp4: B [G][N][K/2] packed E2M1 with 1x32 scales (NT only).
int m_grouped_contiguous(bool b_nmajor, bool fp4, int M_total, int N, int K, int G, const uint8_t* a,
                         const int32_t* sfa, const uint8_t* b, const int32_t* sfb, const int32_t* m_indices,
                         void* d, int d_dtype, fg_stream_t stream) {
    if (M_total < 0 || M_total % 128 != 0 || G < 1) return FG_ERR_INVALID_ARG;
    int rc = check_nt_operands(N, K, a, sfa, b, sfb, d, d_dtype, fp4);
    if (rc) return rc;
    if (!m_indices || !aligned4(m_indices)) return FG_ERR_INVALID_ARG;
    if ((long long)G * N > 0x7fffffffLL) return FG_ERR_INVALID_ARG;
    if (M_total == 0) return FG_OK;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st))) return rc;
    const int sms = sms_in_use(*st);
    const int num_mb = M_total / 128;
    const bool heavy = d_dtype == FG_F32;
    const int bn = b_nmajor ? choose_bn_tn(num_mb, N, sms, heavy) : choose_bn_nt(num_mb, N, sms, heavy, fp4);
    GemmParams p{};
    p.kind = fg::kContiguous;
    p.M = M_total; p.N = N; p.K = K; p.G = G;
    p.d_f32 = d_dtype == FG_F32; p.has_c = 0;
    p.num_mb = num_mb; p.num_nb = ceil_div(N, bn);
    p.sfa = sfa; p.sfb = sfb;
    p.sfa_ld = align4(M_total);
    set_b_scales(p, N, K, fp4);
    p.sfa_rows = M_total;
    p.m_indices = m_indices;
    p.d = d;
    fill_common(p, *st);
    p.b_gstride_k = K;
    fg::GemmMaps gm;
    std::memset(&gm, 0, sizeof(gm));
    CUtensorMap &ma = gm.a, &mb = gm.b;
    const bool b_ok = b_nmajor
        ? encode_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, N, (uint64_t)G * K, N, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B)
        : encode_b_nt(&mb, b, K, (uint64_t)G * N, bn, fp4);
    if (!encode_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, M_total, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !b_ok || !encode_d_maps(gm, d, N, M_total, p.d_f32))
        return FG_ERR_INVALID_ARG;
    const long long tiles = (long long)p.num_mb * p.num_nb;
    const int grid = (int)(tiles < sms ? tiles : sms);
    if (print_configs())
        std::fprintf(stderr, "[fg] m_grouped_%s_contiguous M_total=%d N=%d K=%d G=%d BN=%d grid=%d\n",
                     b_nmajor ? "nn" : (fp4 ? "fp8_fp4_nt" : "nt"), M_total, N, K, G, bn, grid);
    if (b_nmajor) return launch_mn(fg::kMajNN, bn, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
    if (fp4) return launch_fp4(bn, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
    return launch_nt(bn, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
}

// Dense GEMM with an MN-major operand: maj = kMajNN (B [K][N]), kMajTN (A [K][M], B [K][N])
// or kMajTT (A [K][M]).  Same scales, C and D as the NT GEMM.
int dense_mn(int maj, int M, int N, int K, const uint8_t* a, const int32_t* sfa, const uint8_t* b,
             const int32_t* sfb, const float* c, void* d, int d_dtype, fg_stream_t stream) {
    const bool a_mn = (maj & 1) != 0, b_mn = (maj & 2) != 0;
    if (M < 0) return FG_ERR_INVALID_ARG;
    int rc = check_nt_operands(N, K, a, sfa, b, sfb, d, d_dtype);
    if (rc) return rc;
    if (a_mn && M % 16 != 0) return FG_ERR_INVALID_ARG;   // [K][M] rows: 16-byte TMA pitch
    if (c && !aligned16(c)) return FG_ERR_INVALID_ARG;
    if (c && d_dtype != FG_F32) return FG_ERR_UNSUPPORTED;
    if (M == 0) return FG_OK;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st))) return rc;
    const int sms = sms_in_use(*st);
    const int num_mb = ceil_div(M, 128);
    int bn;
    if (b_mn) {
        bn = choose_bn_tn(num_mb, N, sms, c != nullptr || d_dtype == FG_F32);   // whole 128-column atoms of B
    } else {                                                  // K-major B: the NT widths 128/224/256
        const int b0 = choose_bn_nt(num_mb, N, sms, c != nullptr || d_dtype == FG_F32);
        bn = b0 <= 128 ? 128 : (b0 <= 224 ? 224 : 256);
    }
    GemmParams p{};
    fill_common(p, *st);
    p.kind = fg::kDense;
    p.M = M; p.N = N; p.K = K; p.G = 1;
    p.d_f32 = d_dtype == FG_F32; p.has_c = c != nullptr;
    p.c_in_d = c != nullptr && static_cast<const void*>(c) == d;
    p.num_mb = num_mb;
    p.num_nb = ceil_div(N, bn);
    p.sfa = sfa; p.sfb = sfb;
    p.sfa_ld = align4(M); p.sfb_ld = align4(ceil_div(N, 128));
    p.sfa_rows = M;
    p.d = d;
    p.c = c;
    p.a_box_rows = (!a_mn && M <= 64) ? 64 : 128;
    fg::GemmMaps gm;
    std::memset(&gm, 0, sizeof(gm));
    CUtensorMap &ma = gm.a, &mb = gm.b, &mc = gm.c;
    const bool a_ok = a_mn
        ? encode_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, M, K, M, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B)
        : encode_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, M, K, 128, p.a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
    const bool b_ok = b_mn
        ? encode_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, N, K, N, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B)
        : encode_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, K, N, K, 128, bn, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!a_ok || !b_ok || !encode_d_maps(gm, d, N, M, p.d_f32) || (c && !encode_c_maps(gm, c, N, M)))
        return FG_ERR_INVALID_ARG;
    const long long tiles = (long long)p.num_mb * p.num_nb;
    const int grid = (int)(tiles < sms ? tiles : sms);
    if (print_configs())
        std::fprintf(stderr, "[fg] fp8_gemm_%s M=%d N=%d K=%d BN=%d tiles=%lld grid=%d\n",
                     maj == fg::kMajNN ? "nn" : (maj == fg::kMajTN ? "tn" : "tt"), M, N, K, bn, tiles, grid);
    return launch_mn(maj, bn, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int fg_m_grouped_fp8_gemm_nt_contiguous(int M_total, int N, int K, int G, const uint8_t* a,
                                        const int32_t* sfa, const uint8_t* b, const int32_t* sfb,
                                        const int32_t* m_indices, void* d, int d_dtype,
                                        fg_stream_t stream) {
    return m_grouped_contiguous(false, false, M_total, N, K, G, a, sfa, b, sfb, m_indices, d, d_dtype, stream);
}

int fg_m_grouped_fp8_gemm_nn_contiguous(int M_total, int N, int K, int G, const uint8_t* a,
                                        const int32_t* sfa, const uint8_t* b, const int32_t* sfb,
                                        const int32_t* m_indices, void* d, int d_dtype,
                                        fg_stream_t stream) {
    return m_grouped_contiguous(true, false, M_total, N, K, G, a, sfa, b, sfb, m_indices, d, d_dtype, stream);
}

int fg_fp8_gemm_nn(int M, int N, int K, const uint8_t* a, const int32_t* sfa, const uint8_t* b,
                   const int32_t* sfb, const float* c, void* d, int d_dtype, fg_stream_t stream) {
    return dense_mn(fg::kMajNN, M, N, K, a, sfa, b, sfb, c, d, d_dtype, stream);
}

int fg_fp8_gemm_tn(int M, int N, int K, const uint8_t* a, const int32_t* sfa, const uint8_t* b,
                   const int32_t* sfb, const float* c, void* d, int d_dtype, fg_stream_t stream) {
    return dense_mn(fg::kMajTN, M, N, K, a, sfa, b, sfb, c, d, d_dtype, stream);
}

int fg_fp8_gemm_tt(int M, int N, int K, const uint8_t* a, const int32_t* sfa, const uint8_t* b,
                   const int32_t* sfb, const float* c, void* d, int d_dtype, fg_stream_t stream) {
    return dense_mn(fg::kMajTT, M, N, K, a, sfa, b, sfb, c, d, d_dtype, stream);
}

}  // extern "C"

namespace {

// M-grouped masked GEMM; fp4: B [G][N][K/2] packed E2M1 with 1x32 scales.
int m_grouped_masked(bool fp4, int G, int M_max, int N, int K, const uint8_t* a, const int32_t* sfa,
                     const uint8_t* b, const int32_t* sfb, const int32_t* masked_m, int expected_m, void* d,
                     int d_dtype, fg_stream_t stream) {
    if (G < 1 || G > fg::kMaxGroups || M_max < 1) return FG_ERR_INVALID_ARG;
    if ((long long)G * M_max > 0x7fffffffLL || (long long)G * N > 0x7fffffffLL) return FG_ERR_INVALID_ARG;
    int rc = check_nt_operands(N, K, a, sfa, b, sfb, d, d_dtype, fp4);
    if (rc) return rc;
    if (!masked_m || !aligned4(masked_m)) return FG_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st))) return rc;
    const int sms = sms_in_use(*st);
    const int hint = expected_m > 0 ? (expected_m < M_max ? expected_m : M_max) : M_max;
    const int bn = choose_bn_nt((long long)G * ceil_div(hint, 128), N, sms, d_dtype == FG_F32, fp4);
    GemmParams p{};
    p.kind = fg::kMasked;
    p.M = M_max; p.N = N; p.K = K; p.G = G;
    p.d_f32 = d_dtype == FG_F32; p.has_c = 0;
    p.num_mb = ceil_div(M_max, 128); p.num_nb = ceil_div(N, bn);
    p.sfa = sfa; p.sfb = sfb;
    p.sfa_ld = align4(M_max);
    p.sfa_gstride = (long long)ceil_div(K, 512) * p.sfa_ld;
    set_b_scales(p, N, K, fp4);
    p.sfa_rows = M_max;
    p.masked_m = masked_m;
    p.d = d;
    fill_common(p, *st);
    fg::GemmMaps gm;
    std::memset(&gm, 0, sizeof(gm));
    CUtensorMap &ma = gm.a, &mb = gm.b, &mc = gm.c;
    std::memset(&mc, 0, sizeof(mc));
    if (!encode_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, (uint64_t)G * M_max, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_b_nt(&mb, b, K, (uint64_t)G * N, bn, fp4) ||
        !encode_d_maps(gm, d, N, (long long)G * M_max, p.d_f32))
        return FG_ERR_INVALID_ARG;
    const long long tiles = (long long)G * p.num_mb * p.num_nb;   // upper bound
    const int grid = (int)(tiles < sms ? tiles : sms);
    if (print_configs())
        std::fprintf(stderr, "[fg] m_grouped_%smasked G=%d M_max=%d N=%d K=%d BN=%d grid=%d\n",
                     fp4 ? "fp8_fp4_" : "", G, M_max, N, K, bn, grid);
    if (fp4) return launch_fp4(bn, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
    return launch_nt(bn, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int fg_fp8_gemm_nt(int M, int N, int K, const uint8_t* a, const int32_t* sfa, const uint8_t* b,
                   const int32_t* sfb, const float* c, void* d, int d_dtype, fg_stream_t stream) {
    return dense_nt(false, M, N, K, a, sfa, b, sfb, c, d, d_dtype, stream);
}

int fg_fp8_fp4_gemm_nt(int M, int N, int K, const uint8_t* a, const int32_t* sfa, const uint8_t* b,
                       const int32_t* sfb, const float* c, void* d, int d_dtype, fg_stream_t stream) {
    return dense_nt(true, M, N, K, a, sfa, b, sfb, c, d, d_dtype, stream);
}

int fg_m_grouped_fp8_gemm_nt_masked(int G, int M_max, int N, int K, const uint8_t* a,
                                    const int32_t* sfa, const uint8_t* b, const int32_t* sfb,
                                    const int32_t* masked_m, int expected_m, void* d, int d_dtype,
                                    fg_stream_t stream) {
    return m_grouped_masked(false, G, M_max, N, K, a, sfa, b, sfb, masked_m, expected_m, d, d_dtype, stream);
}

int fg_m_grouped_fp8_fp4_gemm_nt_masked(int G, int M_max, int N, int K, const uint8_t* a,
                                        const int32_t* sfa, const uint8_t* b, const int32_t* sfb,
                                        const int32_t* masked_m, int expected_m, void* d, int d_dtype,
                                        fg_stream_t stream) {
    return m_grouped_masked(true, G, M_max, N, K, a, sfa, b, sfb, masked_m, expected_m, d, d_dtype, stream);
}

int fg_m_grouped_fp8_fp4_gemm_nt_contiguous(int M_total, int N, int K, int G, const uint8_t* a,
                                            const int32_t* sfa, const uint8_t* b, const int32_t* sfb,
                                            const int32_t* m_indices, void* d, int d_dtype,
                                            fg_stream_t stream) {
    return m_grouped_contiguous(false, true, M_total, N, K, G, a, sfa, b, sfb, m_indices, d, d_dtype, stream);
}

}  // extern "C"

namespace {

// Gate-up GEMM + SwiGLU + requantisation, contiguous layout; fp4: B [G][2I][K/2] packed
// E2M1 with 1x32 scales.
int swiglu_contiguous(bool fp4, int M_total, int I, int K, int G, const uint8_t* a, const int32_t* sfa,
                      const uint8_t* b, const int32_t* sfb, const int32_t* m_indices, uint8_t* q, int32_t* sfq,
                      fg_stream_t stream) {
    if (M_total < 0 || M_total % 128 != 0 || G < 1 || I < 128 || I % 128 != 0) return FG_ERR_INVALID_ARG;
    const int N = 2 * I;
    int rc = check_nt_operands(N, K, a, sfa, b, sfb, q, FG_BF16, fp4);
    if (rc) return rc;
    if (!sfq || !aligned4(sfq) || !m_indices || !aligned4(m_indices)) return FG_ERR_INVALID_ARG;
    if ((long long)G * N > 0x7fffffffLL) return FG_ERR_INVALID_ARG;
    if (M_total == 0) return FG_OK;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st))) return rc;
    const int sms = sms_in_use(*st);
    GemmParams p{};
    fill_common(p, *st);
    p.kind = fg::kContiguous;
    p.M = M_total; p.N = N; p.K = K; p.G = G;
    p.num_mb = M_total / 128; p.num_nb = I / 128;
    p.sfa = sfa; p.sfb = sfb;
    p.sfa_ld = align4(M_total);
    set_b_scales(p, N, K, fp4);
    p.sfa_rows = M_total;
    p.m_indices = m_indices;
    p.d = q;
    p.sfq = sfq;
    p.sfq_ld = align4(M_total);
    fg::GemmMaps gm;
    std::memset(&gm, 0, sizeof(gm));
    if (!encode_2d(&gm.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, M_total, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_swiglu_b(&gm.b, b, K, I, G, fp4) ||
        !encode_2d(&gm.d, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, I, M_total, I, 128, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return FG_ERR_INVALID_ARG;
    const long long tiles = (long long)p.num_mb * p.num_nb;
    const int grid = (int)(tiles < sms ? tiles : sms);
    if (print_configs())
        std::fprintf(stderr, "[fg] m_grouped_%scontiguous_swiglu M_total=%d I=%d K=%d G=%d grid=%d\n",
                     fp4 ? "fp8_fp4_" : "", M_total, I, K, G, grid);
    return launch_swiglu(fp4, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
}

// The masked layout of swiglu_contiguous.
int swiglu_masked(bool fp4, int G, int M_max, int I, int K, const uint8_t* a, const int32_t* sfa, const uint8_t* b,
                  const int32_t* sfb, const int32_t* masked_m, uint8_t* q, int32_t* sfq, fg_stream_t stream) {
    if (G < 1 || G > fg::kMaxGroups || M_max < 1 || I < 128 || I % 128 != 0) return FG_ERR_INVALID_ARG;
    const int N = 2 * I;
    if ((long long)G * M_max > 0x7fffffffLL || (long long)G * N > 0x7fffffffLL) return FG_ERR_INVALID_ARG;
    int rc = check_nt_operands(N, K, a, sfa, b, sfb, q, FG_BF16, fp4);
    if (rc) return rc;
    if (!sfq || !aligned4(sfq) || !masked_m || !aligned4(masked_m)) return FG_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st))) return rc;
    const int sms = sms_in_use(*st);
    GemmParams p{};
    fill_common(p, *st);
    p.kind = fg::kMasked;
    p.M = M_max; p.N = N; p.K = K; p.G = G;
    p.num_mb = ceil_div(M_max, 128); p.num_nb = I / 128;
    p.sfa = sfa; p.sfb = sfb;
    p.sfa_ld = align4(M_max);
    p.sfa_gstride = (long long)ceil_div(K, 512) * p.sfa_ld;
    set_b_scales(p, N, K, fp4);
    p.sfa_rows = M_max;
    p.masked_m = masked_m;
    p.d = q;
    p.sfq = sfq;
    p.sfq_ld = align4(M_max);
    p.sfq_gstride = (long long)ceil_div(I, 512) * p.sfq_ld;
    fg::GemmMaps gm;
    std::memset(&gm, 0, sizeof(gm));
    if (!encode_2d(&gm.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, (uint64_t)G * M_max, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_swiglu_b(&gm.b, b, K, I, G, fp4) ||
        !encode_2d(&gm.d, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, I, (uint64_t)G * M_max, I, 128, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return FG_ERR_INVALID_ARG;
    const long long tiles = (long long)G * p.num_mb * p.num_nb;   // upper bound
    const int grid = (int)(tiles < sms ? tiles : sms);
    if (print_configs())
        std::fprintf(stderr, "[fg] m_grouped_%smasked_swiglu G=%d M_max=%d I=%d K=%d grid=%d\n",
                     fp4 ? "fp8_fp4_" : "", G, M_max, I, K, grid);
    return launch_swiglu(fp4, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int fg_m_grouped_fp8_gemm_nt_contiguous_swiglu(int M_total, int I, int K, int G, const uint8_t* a,
                                               const int32_t* sfa, const uint8_t* b, const int32_t* sfb,
                                               const int32_t* m_indices, uint8_t* q, int32_t* sfq,
                                               fg_stream_t stream) {
    return swiglu_contiguous(false, M_total, I, K, G, a, sfa, b, sfb, m_indices, q, sfq, stream);
}

int fg_m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(int M_total, int I, int K, int G, const uint8_t* a,
                                                   const int32_t* sfa, const uint8_t* b, const int32_t* sfb,
                                                   const int32_t* m_indices, uint8_t* q, int32_t* sfq,
                                                   fg_stream_t stream) {
    return swiglu_contiguous(true, M_total, I, K, G, a, sfa, b, sfb, m_indices, q, sfq, stream);
}

int fg_m_grouped_fp8_gemm_nt_masked_swiglu(int G, int M_max, int I, int K, const uint8_t* a,
                                           const int32_t* sfa, const uint8_t* b, const int32_t* sfb,
                                           const int32_t* masked_m, uint8_t* q, int32_t* sfq,
                                           fg_stream_t stream) {
    return swiglu_masked(false, G, M_max, I, K, a, sfa, b, sfb, masked_m, q, sfq, stream);
}

int fg_m_grouped_fp8_fp4_gemm_nt_masked_swiglu(int G, int M_max, int I, int K, const uint8_t* a,
                                               const int32_t* sfa, const uint8_t* b, const int32_t* sfb,
                                               const int32_t* masked_m, uint8_t* q, int32_t* sfq,
                                               fg_stream_t stream) {
    return swiglu_masked(true, G, M_max, I, K, a, sfa, b, sfb, masked_m, q, sfq, stream);
}

int fg_fp8_mqa_logits(int S, int T, int H, int D, const uint8_t* q, const uint8_t* kv, const float* kv_sf,
                      const float* weights, const int32_t* ks, const int32_t* ke, int clean_logits, float* out,
                      fg_stream_t stream) {
    if (S < 0 || T < 1 || H < 1 || D < 1) return FG_ERR_INVALID_ARG;
    if (H != 64 || D != 128) return FG_ERR_UNSUPPORTED;
    if ((long long)S * H > 0x7fffffffLL) return FG_ERR_INVALID_ARG;
    if (!q || !kv || !kv_sf || !weights || !ks || !ke || !out) return FG_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned4(kv_sf) || !aligned4(weights) || !aligned4(ks) ||
        !aligned4(ke) || !aligned4(out))
        return FG_ERR_INVALID_ARG;
    if (S == 0) return FG_OK;
    DeviceState* st = nullptr;
    int rc;
    if ((rc = device_state(&st))) return rc;
    const int sms = sms_in_use(*st);
    fg::MqaParams p{};
    p.S = S; p.T = T;
    p.kv_sf = kv_sf; p.weights = weights; p.ks = ks; p.ke = ke; p.out = out;
    p.clean = clean_logits ? 1 : 0;
    p.status = st->status;
    p.timeout_ns = g_timeout_ns;
    p.pdl = g_pdl;
    fg::MqaMaps mm;
    std::memset(&mm, 0, sizeof(mm));
    if (!encode_2d(&mm.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, 128, (uint64_t)S * 64, 128, 128, fg::kMqaTokens * 64,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&mm.kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, kv, 128, (uint64_t)T, 128, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return FG_ERR_INVALID_ARG;
    const int groups = (S + fg::kMqaTokens - 1) / fg::kMqaTokens;
    const int grid = groups < sms ? groups : sms;
    if (print_configs())
        std::fprintf(stderr, "[fg] fp8_mqa_logits S=%d T=%d H=%d D=%d clean=%d grid=%d\n", S, T, H, D, p.clean, grid);
    if (fg::launch_mqa(p, mm, grid, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FG_ERR_CUDA;
    }
    return FG_OK;
}

int fg_k_grouped_fp8_gemm_tn_contiguous(int G, int M, int N, int K_total, const uint8_t* a,
                                        const int32_t* sfa, const uint8_t* b, const int32_t* sfb,
                                        const int32_t* ks, const float* c, float* d,
                                        fg_stream_t stream) {
    if (G < 1 || G > fg::kMaxGroups || M < 16 || M % 16 != 0 || N < 16 || N % 16 != 0 ||
        K_total < 0 || K_total % 128 != 0)
        return FG_ERR_INVALID_ARG;
    if ((long long)G * M > 0x7fffffffLL) return FG_ERR_INVALID_ARG;
    if (!ks || !aligned4(ks) || !d || !aligned16(d) || (c && !aligned16(c))) return FG_ERR_INVALID_ARG;
    if (K_total > 0 && (!a || !sfa || !b || !sfb || !aligned16(a) || !aligned16(sfa) ||
                        !aligned16(b) || !aligned16(sfb)))
        return FG_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc;
    if ((rc = device_state(&st))) return rc;
    const int sms = sms_in_use(*st);
    const int num_mb = ceil_div(M, 128);
    const int bn = choose_bn_tn((long long)G * num_mb, N, sms, true);
    GemmParams p{};
    p.kind = fg::kKGrouped;
    p.M = M; p.N = N; p.K = K_total; p.G = G;
    p.d_f32 = 1; p.has_c = c != nullptr;
    p.c_in_d = c != nullptr && c == d;
    p.c = c;
    p.num_mb = num_mb; p.num_nb = ceil_div(N, bn);
    p.sfa = sfa; p.sfb = sfb;
    p.sfa_ld = align4(M); p.sfb_ld = align4(N);
    p.sfb_per_row = 1;
    p.sfa_rows = M;
    p.ks = ks;
    p.d = d;
    fill_common(p, *st);
    fg::GemmMaps gm;
    std::memset(&gm, 0, sizeof(gm));
    CUtensorMap &ma = gm.a, &mb = gm.b, &mc = gm.c, &md = gm.d;
    std::memset(&ma, 0, sizeof(ma));
    std::memset(&mb, 0, sizeof(mb));
    std::memset(&mc, 0, sizeof(mc));
    // C and D as [G][M][N]: boxes never cross into the next group's rows.
    const uint64_t pitch1 = (uint64_t)N * 4, pitch2 = (uint64_t)M * N * 4;
    if (!encode_3d(&md, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, d, N, M, G, pitch1, pitch2, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B) ||
        (c && !encode_3d(&mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, c, N, M, G, pitch1, pitch2, 32, 32,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
        return FG_ERR_INVALID_ARG;

    // With K_total == 0 every segment is empty and no operand load is ever issued.
    if (K_total > 0 &&
        (!encode_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, M, K_total, M, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
         !encode_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, N, K_total, N, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B)))
        return FG_ERR_INVALID_ARG;
    const long long tiles = (long long)G * p.num_mb * p.num_nb;
    const int grid = (int)(tiles < sms ? tiles : sms);
    if (print_configs())
        std::fprintf(stderr, "[fg] k_grouped_tn G=%d M=%d N=%d K_total=%d BN=%d grid=%d\n", G, M, N, K_total, bn, grid);
    return launch_mn(fg::kMajTN, bn, p, gm, grid, reinterpret_cast<cudaStream_t>(stream));
}

int fg_get_mk_alignment_for_contiguous_layout(void) { return 128; }

int fg_get_tma_aligned_size(int x, int elem_bytes) {
    if (x < 0 || (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)) return -1;
    const int per = 16 / elem_bytes;
    return (x + per - 1) / per * per;
}

void fg_set_num_sms(int n) {
    std::lock_guard<std::mutex> lock(g_mu);
    g_num_sms_limit = n > 0 ? n : 0;
}

void fg_set_pdl(int enable) {
    std::lock_guard<std::mutex> lock(g_mu);
    g_pdl = enable ? 1 : 0;
}

int fg_get_pdl(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    return g_pdl;
}

int fg_get_num_sms(void) {
    DeviceState* st = nullptr;
    if (device_state(&st)) return -1;
    return sms_in_use(*st);
}

int fg_get_device_error(fg_stream_t stream, int* detail) {
    if (detail) *detail = 0;
    DeviceState* st = nullptr;
    if (device_state(&st)) return FG_ERR_CUDA;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    {
        std::lock_guard<std::mutex> lock(g_take_mu);
        take_status_kernel<<<1, 1, 0, s>>>(st->status, st->taken);
        if (cudaGetLastError() != cudaSuccess ||
            cudaMemcpyAsync(&v, st->taken, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess) {
            cudaGetLastError();
            return FG_ERR_CUDA;
        }
    }
    if (detail) *detail = v;
    if (v == 0) return FG_OK;
    if (v & fg::kErrTimeout) return FG_ERR_DEVICE_TIMEOUT;
    return FG_ERR_DEVICE_CONTRACT;
}

const char* fg_status_string(int status) {
    switch (status) {
        case FG_OK: return "ok";
        case FG_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer, bad shape or dtype)";
        case FG_ERR_UNSUPPORTED: return "unsupported combination (e.g. C with a BF16 D)";
        case FG_ERR_CUDA: return "CUDA runtime or driver call failed";
        case FG_ERR_DEVICE_CONTRACT: return "device-side contract violation (indices, mask or K segments)";
        case FG_ERR_DEVICE_TIMEOUT: return "bounded wait inside a kernel timed out";
        default: return "unknown status";
    }
}

void fg_debug_inject_stall(int enable, uint32_t timeout_us) {
    std::lock_guard<std::mutex> lock(g_mu);
    g_debug_stall = enable ? 1 : 0;
    g_timeout_ns = enable && timeout_us > 0 ? 1000ull * timeout_us : kDefaultTimeoutNs;
}

}  // extern "C"
