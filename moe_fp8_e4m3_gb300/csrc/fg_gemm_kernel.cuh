// fg_gemm_kernel.cuh - persistent, warp-specialised, block-scaled FP8 GEMM for sm_103a.
//
// One kernel template covers the four GEMMs of the DeepGEMM pages ("DeepGEMM
// Documentation", section 4 "Understand DeepGEMM GEMM Naming and Layouts" and section 9
// "Use Normal and Grouped GEMM Kernels"): dense NT, M-grouped contiguous NT, M-grouped
// masked NT and K-grouped contiguous TN.
//
// Per output tile (128 rows x BN columns) and per 128-wide K-group g the kernel forms
//     acc[m, n] += sa[m, g] * sb[n, g] * sum_{k in g} a[m, k] * b[n, k]
// with tcgen05.mma kind::mxf8f6f4 block_scale: the UE8M0 scales are applied inside the
// tensor core and the FP32 accumulator lives in tensor memory (TMEM) for the whole K
// loop, so every partial sum is promoted to FP32 with its scale already applied (the
// pages' "two-level accumulation", Deepseek AI Libera DeepGEMM article, section
// "Details and technical benefits", realised by the hardware's scaled MMA instead of a
// CUDA-core FMA pass).  A packed UE8M0 word holds the scales of four consecutive
// K-groups; it is copied to TMEM unchanged and the MMA's scale-factor byte selector
// picks byte (g mod 4).
//
// FP8 x FP4 (operand-major bit 2): B holds E2M1 codes, two per byte, with one UE8M0 scale
// per 32 K elements of a row.  The tensor map unpacks B into the padded shared-memory form
// of a sub-byte MMA operand (the same bytes per stage as E4M3 B), the instruction
// descriptor names E2M1 for B, B's scale word changes every K-group (its four bytes are
// the K-group's four 32-wide blocks), and each K=32 MMA selects its own B byte.
//
// Warp roles (320 threads):
//   warps 0, 8  TMA producers of A tiles into a ring of shared-memory stages (even / odd
//               stages)
//   warp 1      TMEM owner + MMA issuer (one elected lane)
//   warps 2, 9  TMA producers of B tiles (even / odd stages).  Measured on GB300: the TMA
//               loads one warp issues complete one after another, about 0.34 us each
//               from L2 whatever the box size (4-32 KB), while loads of different warps
//               proceed in parallel; so each operand streams from two warps.
//   warp 3      scale loader: the packed UE8M0 words of each tile (one word row per four
//               K-groups), copied by the whole warp with 4-byte cp.async straight into the
//               tcgen05.cp 32x4 atom layout of the stage that starts the word row; every lane
//               arrives on every stage's full barrier once its copies have landed, so the MMA
//               issuer waits once per stage for operands and scales, and this warp never
//               waits for load latency
//   warps 4..7  epilogue: TMEM -> registers, + C -> BF16/FP32 -> TMA store, each warp on
//               its own 32 rows.  A C that is an array of its own (the kSepC variants) lands
//               in C slots, loaded ahead by lane 0 and refilled as soon as read; D chunks
//               leave from store slots through TMA stores issued by lane 1 (the two TMA
//               streams of a warp proceed side by side).  When D is C itself (in-place
//               accumulation) no C is loaded: the accumulator chunk leaves through a TMA
//               reduce-add, and L2 adds it onto D.
// The MMA issuer's loop is lean (measured on GB300: ~55 clocks to issue one tcgen05.mma and
// ~200 to test an mbarrier, against 448 clocks of tensor work per 128 x 224 x 128 K-group):
// descriptors are precomputed per stage, and when the next two stages have both landed (two
// pipelined non-blocking tests) it issues both stages' MMAs after one round of waiting.
// The mainloop's pace is the ring's round trip (load latency + MMA issue and execution)
// over its stage count, so shared memory goes to stages first.
// Accumulators are double-buffered in TMEM when two fit next to the scale slots
// (BN <= 224), so the epilogue of one tile overlaps the MMAs of the next.
// Each variant serves one layout (dense, contiguous, masked, K-grouped), fixed at compile
// time, so a launch fetches one tile walk's code.
//
// Split-K clusters (dense NT, few output tiles): a cluster of `split` CTAs shares one
// output tile, each CTA runs a contiguous share of the K-groups, and the partial FP32
// tiles are summed through distributed shared memory in rank order (deterministic),
// each CTA reducing and storing one slice of the tile's columns.
// Every role walks the same static persistent tile sequence (tile = blockIdx.x +
// i * gridDim.x), decoded from device-resident segment data without host sync.
//
// Every wait is bounded (globaltimer); on expiry the CTA records a time-out in the
// device status word, raises a shared abort flag that every other wait observes,
// drains its own in-flight tensor-core work and TMA copies (again bounded), frees TMEM
// and returns.  Nothing traps.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "fg_fp8.cuh"
#include "fg_ptx.cuh"

namespace fg {

enum GemmKind : int { kDense = 0, kContiguous = 1, kMasked = 2, kKGrouped = 3 };

// Operand majors of a kernel variant (the pages' layout letters, D = C + A @ B):
// bit 0 set = A stored [K][M] (M-major, "T"), clear = [M][K] (K-major, "N");
// bit 1 set = B stored [K][N] (N-major, "N"), clear = [N][K] (K-major, "T");
// bit 2 set = B holds FP4 (E2M1) codes, two per byte along K, with one UE8M0 scale per
// 32 K elements of each row (the FP8 x FP4 GEMM; K-major B only).
enum : int { kMajNT = 0, kMajTT = 1, kMajNN = 2, kMajTN = 3, kMajNTF4 = 4 };

// Device status codes (the word keeps the first event).
enum : int {
    kErrContract = 0x100,      // | check id
    kErrTimeout = 0x200,       // | where
    kChkGroupIndex = 1,        // m_indices names a group >= G
    kChkMixedBlock = 2,        // a row names another group than its block
    kChkMaskRange = 3,         // masked_m outside [0, M_max]
    kChkKSegments = 4,         // ks not multiples of 128 / negative / wrong sum
    kChkSplit = 5,             // split-K launch without one tile per cluster
    kWaitProducer = 1, kWaitMma = 2, kWaitScales = 3, kWaitEpilogue = 4, kWaitDrain = 5,
    kWaitEpilogueC = 6, kWaitExchange = 7, kWaitScaleSlot = 8, kWaitProducerB = 9, kWaitEpilogueSync = 10,
    kWaitEpilogueCFree = 11,
};

constexpr int kMaxGroups = 256;   // masked / K-grouped groups held in shared memory
constexpr int kSmemLimit = 232448;
constexpr int kGemmThreads = 320;
constexpr int kEpiWarp0 = 4;      // first epilogue warp
constexpr int kEpiThread0 = 32 * kEpiWarp0;

// Tensor maps of one launch (a kernel parameter, so the TMA unit reads them from
// parameter space): A and B operand tiles, C and D in 32-row x 128-byte boxes (one epilogue
// warp's chunk).
struct GemmMaps {
    CUtensorMap a, b, c, d;
};

struct GemmParams {
    int kind;
    int M, N, K;           // dense M,N,K | contiguous M_total | masked M_max | K-grouped M,N,K_total
    int G;
    int d_f32, has_c;
    int c_in_d;            // C is D itself (in-place accumulation): D += A @ B by TMA reduce-add
    int prefetch_b;        // dense, one tile per CTA: prefetch the tile's B into L2 before the
                           // grid-dependency wait
    int num_mb, num_nb;    // tile grid of one group
    const int32_t* sfa;
    const int32_t* sfb;
    int sfa_ld, sfb_ld;    // int32 words per packed-word row of the scale arrays
    long long sfa_gstride, sfb_gstride;  // words between groups (masked SFA, grouped SFB)
    int sfa_rows;          // MN extent of the SFA rows
    const int32_t* m_indices;
    const int32_t* masked_m;
    const int32_t* ks;
    void* d;               // for the per-thread store path (partially valid row groups)
    const float* c;        // C for the split-K reduction (nullable)
    int split;             // CTAs per cluster sharing one tile along K (1: no split)
    int a_box_rows;        // rows of the A tensor-map box (128, or 64 when every tile has <= 64 rows)
    int pdl;               // host side: launch with programmatic stream serialisation
    int sfb_per_row;       // B scales: one per row of B and 1x128 K-group (else one per 128x128 block)
    int32_t* sfq;          // SwiGLU epilogue: packed scale words of the quantised output
    int sfq_ld;            //   int32 words per packed-word row (align4 of its rows)
    long long sfq_gstride; //   words between groups (masked layout)
    long long b_gstride_k; // MN-major grouped B: rows of the [G*K][N] map between groups (K)
    int* status;
    unsigned long long timeout_ns;
    int debug_stall;
};

template <int BN, bool kSplit = false, bool kSwiGLU = false, bool kSepC = false>
struct TileCfg {
    static constexpr int kBM = 128, kBK = 128;
    static constexpr int kSfbAtoms = (BN + 127) / 128;
    static constexpr int kSfCols = 4 + 4 * kSfbAtoms;    // TMEM columns of one scale slot
    static constexpr int kNumAcc = (2 * BN + 32 <= 512) ? 2 : 1;
    static constexpr int kSfCol0 = (kNumAcc * BN + 15) / 16 * 16;
    static_assert(kSfCol0 + 16 + kSfCols <= 512, "TMEM columns");
    static constexpr int kABytes = kBM * kBK;              // 16 KB
    static constexpr int kBBytes = BN * kBK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    // Scale words of a stage (used by the stages that start a packed word row, four
    // K-groups): the 128 A rows' words and the words of the BN B rows, each as 32x4 atoms of
    // 512 bytes.
    static constexpr int kSfaBytes = 512;
    static constexpr int kSfbBytes = kSfbAtoms * 512;
    static constexpr int kSfSlotBytes = kSfaBytes + kSfbBytes;
    // Epilogue, per warp: kCSlots slots where C chunks land (refilled as soon as read) and
    // kDSlots slots from which D chunks are stored; each slot is 32 rows x 128 bytes (one
    // chunk: 32 FP32 or 64 BF16 columns).  Only the kSepC variants, launched when C is an
    // array of its own, have C slots: without C, or with D aliasing C (accumulated by a TMA
    // reduce-add), the space goes to pipeline stages.  Split-K variants exchange through
    // the operand ring and use no slots; the SwiGLU variant stages one chunk of codes; tiles
    // too wide for two accumulators give the space to stages even with a separate C (it
    // then lands in the store slot).
    // (measured on GB300: the mainloop of these kernels is bound by the bytes its ring holds
    // in flight, so every stage that fits counts)
    // The stages are sized with one store slot per warp; a second one (the store of one chunk
    // overlapping the next chunk's work) is added where the space left over holds it.
    // BN 192/224 keep one C slot, which leaves room for a fourth stage: measured on GB300 on
    // 4096 x 7168 x 2048 with a separate FP32 C, 4 stages with 1 C slot and 1 store slot ran
    // 70.8 us, 3 stages with 3 C slots and 2 store slots 72.4 us, and 4 stages with C landing
    // in the store slots (no prefetch) 91.2 us.  Below 192 one C slot would not free a stage.
    static constexpr int kCSlots = (!kSepC || kSplit || kSwiGLU) ? 0 : (BN >= 256 ? 0 : (BN >= 192 ? 1 : 2));
    static constexpr int kSlotBytes = 4096;
    static constexpr int kDSlotsMin = kSplit ? 0 : 1;
    static constexpr int kEpiMin = 4 * (kCSlots + kDSlotsMin) * kSlotBytes;
    static constexpr int kMiscBytes = 1024 + 2 * (kMaxGroups + 1) * 4;   // barriers etc. + group tables
    static constexpr int kStages0 = (kSmemLimit - 1024 - kEpiMin - kMiscBytes) / (kStageBytes + kSfSlotBytes);
    static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
    static constexpr int kSpare = kSmemLimit - 1024 - kEpiMin - kMiscBytes - kStages * (kStageBytes + kSfSlotBytes);
    static constexpr int kDSlots = (kSplit || kSwiGLU) ? kDSlotsMin : (kSpare >= 4 * kSlotBytes ? 2 : 1);
    static constexpr int kEpiBytes = 4 * (kCSlots + kDSlots) * kSlotBytes;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kABytes;
    static constexpr int kOffEpi = kOffB + kStages * kBBytes;                 // 1024-aligned
    static constexpr int kOffCSlots = kOffEpi;
    static constexpr int kOffDSlots = kOffEpi + 4 * kCSlots * kSlotBytes;
    static constexpr int kOffSf = kOffEpi + kEpiBytes;
    static constexpr int kOffBar = kOffSf + kStages * kSfSlotBytes;
    // per epilogue warp: C landed in one of its C slots / in one of its store slots
    static constexpr int kNumCBars = 4 * (kCSlots + kDSlots);
    static constexpr int kNumBars = 2 * kStages + 2 * kNumAcc + 1 + kNumCBars + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;                   // tmem addr, abort flag, row flags
    static constexpr int kOffSched = kOffMisc + 32;                           // int[kMaxGroups + 1]
    static constexpr int kOffCnt = kOffSched + (kMaxGroups + 1) * 4;
    static constexpr int kSmemBytes = kOffCnt + kMaxGroups * 4 + 1024;       // + alignment slack
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "UMMA N for M=128 (and 32-column chunks)");
    static_assert(kStages >= 2, "pipeline depth");
    static_assert(kNumBars * 8 <= 1024 - 32, "barrier area");
    static_assert(kSmemBytes <= kSmemLimit, "shared memory");
    static_assert(kOffSf % 512 == 0 && kSfSlotBytes % 512 == 0, "scale atoms 512-byte aligned");
    // Split-K exchange buffer: the FP32 partial tile, rows padded by 16 bytes, in the
    // operand ring (idle once the cluster's single tile has been accumulated).
    static constexpr int kXStride = BN + 4;
    static_assert(!kSplit || kStages * (kABytes + kBBytes) >= kBM * kXStride * 4, "split-K exchange buffer");
};

struct Tile {
    int g, n0;
    int a_coord, b_coord;   // NT: rows in the A/B maps; TN: columns (m0 / n0)
    int kb0, nkb;           // first global K-group and number of K-groups
    long long b_krow;       // MN-major B: map row of the tile's K = 0 (group offset)
    int valid_rows;         // rows [0, valid_rows) of the tile lie inside the problem
    long long d_row;        // row of D (flat [rows][N] view) that holds the tile's row 0
    int d_y, d_z;           // coordinates of row 0 in the C/D tensor maps
    int sfa_g, sfa_row;
    bool skip;
};

__device__ __forceinline__ void record_status(int* status, int code) {
    atomicCAS(status, 0, code);
}

struct WaitCtl {
    volatile int* abort;
    int* status;
    unsigned long long timeout_ns;
};

// Bounded mbarrier wait.  Returns false if the CTA is aborting (flag raised here or
// by another role).
// kSleep: a waiting thread sleeps (suspend-time hint) instead of spinning.  Measured on
// GB300: the GEMM gains (its spinning producer and MMA warps share schedulers with the
// epilogue), the MQA kernel loses (its epilogue warps wake later) and spins.
template <bool kCluster = false, bool kSleep = true>
__device__ __forceinline__ bool try_wait_scoped(uint32_t bar, uint32_t parity) {
    if (kCluster) return mbar_try_wait_cluster(bar, parity);
    return kSleep ? mbar_try_wait_sleep(bar, parity) : mbar_try_wait(bar, parity);
}
// kCluster: the barrier is also arrived on from another CTA of the cluster (acquire at
// cluster scope).
template <bool kCluster = false, bool kSleep = true>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtl& w, int where) {
    if (try_wait_scoped<kCluster, kSleep>(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (try_wait_scoped<kCluster, kSleep>(bar, parity)) return true;
        // a spinning wait polls the abort flag and the clock every 32nd round only: each
        // poll is a shared-memory load competing with the tensor cores' operand reads
        if (!kSleep && (it & 31u)) continue;
        if (*w.abort) return false;
        if (globaltimer_ns() - t0 > w.timeout_ns) {
            *w.abort = 1;
            record_status(w.status, kErrTimeout | where);
            return false;
        }
    }
}

// Wait without abort observation, for draining in-flight copies on the way out.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < limit_ns) {
    }
}

// rank: this CTA's rank in its split-K cluster (its share of the K-groups).
// scan: the caller is a whole warp walking the tiles together (the scale loader); it
// checks that a contiguous block whose first row is padding (-1) names no group in any
// later row (such a block is skipped, so its rows would silently stay unwritten).
template <int BN>
__device__ __forceinline__ Tile decode_tile(const GemmParams& p, int kind, int t, const int* sched,
                                            const int* cnt, int& cursor, int rank, int split,
                                            bool scan) {
    Tile tl;
    tl.skip = false;
    tl.g = 0;
    tl.kb0 = 0;
    tl.nkb = p.K / 128;
    tl.sfa_g = 0;
    tl.d_z = 0;
    tl.b_krow = 0;
    if (kind == kDense) {
        const int mb = t % p.num_mb, nb = t / p.num_mb;
        tl.n0 = nb * BN;
        tl.a_coord = mb * 128;
        tl.b_coord = tl.n0;
        tl.valid_rows = min(128, p.M - mb * 128);
        tl.d_row = mb * 128;
        tl.sfa_row = mb * 128;
        if (split > 1) {     // this CTA's share of the K-groups: [r*nkb/split, (r+1)*nkb/split)
            const int nkb = tl.nkb;
            tl.kb0 = rank * nkb / split;
            tl.nkb = (rank + 1) * nkb / split - tl.kb0;
        }
    } else if (kind == kContiguous) {
        const int mb = t / p.num_nb, nb = t % p.num_nb;
        const int g = __ldg(p.m_indices + (long long)mb * 128);
        tl.n0 = nb * BN;
        if (scan && g < 0) {
            const int lane = threadIdx.x & 31;
            const int32_t* blk = p.m_indices + (long long)mb * 128;
            bool named = false;
#pragma unroll
            for (int j = 0; j < 4; ++j) named |= __ldg(blk + lane + 32 * j) >= 0;
            if (__any_sync(0xffffffffu, named) && lane == 0) record_status(p.status, kErrContract | kChkMixedBlock);
        }
        if (g < 0 || g >= p.G) {
            if (g >= p.G) record_status(p.status, kErrContract | kChkGroupIndex);
            tl.skip = true;
        }
        tl.g = (g < 0 || g >= p.G) ? 0 : g;
        tl.a_coord = mb * 128;
        tl.b_coord = tl.g * p.N + tl.n0;
        tl.b_krow = tl.g * p.b_gstride_k;
        tl.valid_rows = 128;
        tl.d_row = (long long)mb * 128;
        tl.sfa_row = mb * 128;
    } else if (kind == kMasked) {
        while (cursor + 1 < p.G && sched[cursor + 1] <= t) ++cursor;
        const int g = cursor;
        const int local = t - sched[g];
        const int mb = local / p.num_nb, nb = local % p.num_nb;
        tl.g = g;
        tl.n0 = nb * BN;
        tl.a_coord = g * p.M + mb * 128;
        tl.b_coord = g * p.N + tl.n0;
        tl.valid_rows = min(128, cnt[g] - mb * 128);
        tl.d_row = (long long)g * p.M + mb * 128;
        tl.sfa_g = g;
        tl.sfa_row = mb * 128;
    } else {  // K-grouped
        const int per_g = p.num_mb * p.num_nb;
        const int g = t / per_g, local = t % per_g;
        const int mb = local / p.num_nb, nb = local % p.num_nb;
        tl.g = g;
        tl.n0 = nb * BN;
        tl.a_coord = mb * 128;
        tl.b_coord = tl.n0;
        tl.kb0 = sched[g];
        tl.nkb = sched[g + 1] - sched[g];
        tl.valid_rows = min(128, p.M - mb * 128);
        tl.d_row = (long long)g * p.M + mb * 128;
        tl.d_y = mb * 128;
        tl.d_z = g;
        tl.sfa_row = mb * 128;
        return tl;
    }
    tl.d_y = static_cast<int>(tl.d_row);
    return tl;
}

// Walks the tiles of one CTA, skipping the ones no role works on.
template <int BN>
struct TileIter {
    int t;
    int cursor;
    int stride;
    int rank;
    int split;
    int kind;
    __device__ __forceinline__ bool next(const GemmParams& p, int total, const int* sched, const int* cnt,
                                         Tile& tl, bool scan = false) {
        while (t < total) {
            tl = decode_tile<BN>(p, kind, t, sched, cnt, cursor, rank, split, scan);
            t += stride;
            if (!tl.skip) return true;
        }
        return false;
    }
};

// Tiles of this CTA: blockIdx.x + i * gridDim.x, or per split-K cluster when clusters share
// tiles.  `kind` is the call's layout (a constant in the dense-only variants, so their
// tile walk compiles to the dense case alone).
template <int BN>
__device__ __forceinline__ TileIter<BN> tiles_of_cta(int rank, int split, int kind) {
    return TileIter<BN>{static_cast<int>(blockIdx.x) / split, 0, static_cast<int>(gridDim.x) / split, rank, split, kind};
}

// ------------------------------------------------------------ split-K exchange
// Epilogue of one tile shared by a split-K cluster (kept out of line: the common
// epilogue path never fetches its code).
//   1. the partial tile (TMEM) -> this CTA's exchange buffer, valid rows only;
//   2. every epilogue warp of the cluster arrives on every CTA's exchange barrier;
//   3. this CTA sums its column slice over the cluster's buffers in rank order
//      (rank 0's value, + rank 1's, ...), adds C and stores D.
// The teardown cluster barrier keeps each buffer alive until every peer has read it.
// Returns false on abort (time-out).
struct SplitTile {
    int valid_rows, n0, N, nkb;
    long long d_row;
    int has_c, d_f32;
    const float* c;
    void* d;
};

template <int BN, class C>
__device__ __noinline__ bool split_k_tile(const SplitTile st, float* xb, uint32_t tmem_acc, uint32_t accf,
                                          uint32_t acc_ph, uint32_t acce, uint32_t xfull, uint32_t x_ph,
                                          const WaitCtl wctl, int rank, int split) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;                                // TMEM sub-partition of this warp
    const int row = q * 32 + lane;
    const int te = static_cast<int>(threadIdx.x) - 32 * kEpiWarp0;   // 0..127 over the epilogue warps
    constexpr int kB = 4;                                  // slice items (float4 groups) per thread and pass
    const int vr = st.valid_rows;
    const int w = BN / split;
    const int col0 = rank * w;
    const int g4 = max(0, min(w, min(BN, st.N - st.n0) - col0)) >> 2;   // float4 groups in the slice
    const int items = vr * g4;
    // C of the slice: every row prefetched into L2 now, the first pass loaded into registers,
    // both while the tile accumulates
    if (st.has_c && te < vr && g4 > 0)
        prefetch_l2_bulk(st.c + (st.d_row + te) * st.N + st.n0 + col0, static_cast<uint32_t>(g4) * 16u);
    float4 cv[kB];
    long long gofs[kB];
    uint32_t xofs[kB];
    auto locate = [&](int u0) {
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int u = u0 + b * 128 + te;
            const int rr = u < items ? u / g4 : 0;
            const int cc = u < items ? col0 + 4 * (u - rr * g4) : 0;
            gofs[b] = (st.d_row + rr) * st.N + st.n0 + cc;
            xofs[b] = static_cast<uint32_t>(rr * C::kXStride + cc) * 4u;
            cv[b] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (u < items && st.has_c) cv[b] = *reinterpret_cast<const float4*>(st.c + gofs[b]);
        }
    };
    locate(0);
    const bool ok = wait_bar(accf, acc_ph, wctl, kWaitEpilogue);
    if (!__all_sync(0xffffffffu, ok)) return false;
    tc_fence_after();
    fence_proxy_async_smem();   // the ring was last used by TMA and the tensor cores
    if (q * 32 < vr) {
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t r[32];
            if (st.nkb > 0) {
                tmem_ld_32x32b_x32(tmem_acc + (static_cast<uint32_t>(q * 32) << 16) + c0, r);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = 0u;
            }
            if (row < vr) {
                float4* dst = reinterpret_cast<float4*>(xb + row * C::kXStride + c0);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                         __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
        mbar_arrive(acce);
        for (int r2 = 0; r2 < split; ++r2) mbar_arrive_remote(map_shared_rank(xfull, r2));
    }
    const bool okx = wait_bar<true>(xfull, x_ph, wctl, kWaitExchange);
    if (!__all_sync(0xffffffffu, okx)) return false;
    const uint32_t xb_u32 = smem_u32(xb);
    for (int u0 = 0; u0 < items; u0 += 128 * kB) {
        if (u0 > 0) locate(u0);
        float4 v[kB];
        for (int r2 = 0; r2 < split; ++r2) {
            const uint32_t base = map_shared_rank(xb_u32, r2);
            float4 x[kB];
#pragma unroll
            for (int b = 0; b < kB; ++b)
                x[b] = (u0 + b * 128 + te < items) ? ld_dsmem_f32x4(base + xofs[b]) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                if (r2 == 0) {
                    v[b] = x[b];
                } else {
                    v[b].x += x[b].x; v[b].y += x[b].y; v[b].z += x[b].z; v[b].w += x[b].w;
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            if (u0 + b * 128 + te >= items) continue;
            const float4 o = make_float4(v[b].x + cv[b].x, v[b].y + cv[b].y, v[b].z + cv[b].z, v[b].w + cv[b].w);
            if (st.d_f32) {
                *reinterpret_cast<float4*>(static_cast<float*>(st.d) + gofs[b]) = o;
            } else {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(o.z, o.w);
                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(st.d) + gofs[b]) =
                    make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
            }
        }
    }
    return true;
}

// SwiGLU variant (kSwiGLU): B holds each group's gate rows [0, N/2) and up rows
// [N/2, N); output column block nb (128 wide) reads gate rows nb*128.. and up rows
// N/2 + nb*128.. into one 256-row B tile, so the accumulator holds gate in columns
// 0..127 and up in 128..255 of the same 128 outputs.  Returns the B-tile row of
// tile row 0 of half h.
__device__ __forceinline__ int swiglu_b_row(const GemmParams& p, const Tile& tl, int h) {
    const int nb = tl.n0 / 256;
    return (tl.b_coord - tl.n0) + (h ? p.N / 2 : 0) + nb * 128;
}

// SiLU(gate) * up of two FP32 accumulator words.  The fast division (<= 2 ulp) keeps
// the epilogue short: the correctly rounded one took ~2x the whole GEMM's time; both are
// far inside one E4M3 spacing of the requantised result.
__device__ __forceinline__ float swiglu_value(uint32_t gate, uint32_t up) {
    const float x = __uint_as_float(gate);
    return __fdividef(x, 1.0f + __expf(-x)) * __uint_as_float(up);
}

template <int BN, int kMaj, bool kSplit, bool kSwiGLU, bool kSepC, int kKindT>
__global__ void __launch_bounds__(kGemmThreads, 1)
fg_gemm_kernel(const GemmParams p, const __grid_constant__ GemmMaps maps) {
    const CUtensorMap& tm_a = maps.a;
    const CUtensorMap& tm_b = maps.b;
    const CUtensorMap& tm_c = maps.c;
    const CUtensorMap& tm_d = maps.d;
    constexpr bool kAmn = (kMaj & 1) != 0, kBmn = (kMaj & 2) != 0;
    // FP4 B: the tensor map unpacks every 16 codes (8 bytes) into a 16-byte shared-memory
    // chunk (the second 8 bytes are padding), so a 128-code K-group row takes the 128 bytes
    // an E4M3 row takes and the MMA walks the stage exactly as for FP8 B; the instruction
    // descriptor names E2M1 for B, and each K=32 MMA selects its own scale byte.
    constexpr bool kFp4B = (kMaj & 4) != 0;
    static_assert(!kFp4B || kMaj == kMajNTF4, "FP4 B is a K-major NT operand");
    static_assert(!(kSplit && (kMaj & 3) != kMajNT), "split-K clusters are a dense NT variant");
    static_assert(!kBmn || BN % 128 == 0, "N-major B tiles are whole 128-column swizzle atoms");
    static_assert(!kSwiGLU || (BN == 256 && (kMaj & 3) == kMajNT && !kSplit),
                  "the SwiGLU epilogue pairs 128 gate and 128 up columns in one NT tile");
    static_assert(!kSepC || (!kSplit && !kSwiGLU), "C slots belong to the plain epilogue");
    static_assert(!kSwiGLU || kKindT == kContiguous || kKindT == kMasked, "the SwiGLU epilogue is an M-grouped layout");
    static_assert(!kSplit || kKindT == kDense, "split-K clusters are dense");
    using C = TileCfg<BN, kSplit, kSwiGLU, kSepC>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Split-K cluster: rank r runs the r-th share of the K-groups.
    const int split = kSplit ? p.split : 1;   // a compile-time 1 outside the split-K variant
    // The layout is fixed at compile time (kKindT; -1 reads it from the call): each variant's
    // code holds one tile walk, so less of it has to be fetched cold when the kernel starts
    // (measured on GB300: the decode GEMM behind the prefill 21.9 -> 19.8 us, the prefill
    // 75.2 -> 72.7 us).
    const int kind = kKindT >= 0 ? kKindT : p.kind;
    const int rank = split > 1 ? static_cast<int>(cluster_ctarank()) : 0;

    const uint32_t bar0 = sbase + C::kOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * C::kStages + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * C::kStages + C::kNumAcc + b); };
    const uint32_t mma_drain_bar = bar0 + 8u * (2 * C::kStages + 2 * C::kNumAcc);
    // epilogue slot barriers of warp ew: C landed in its C slot i / in its store slot j
    const uint32_t ebar0 = bar0 + 8u * (2 * C::kStages + 2 * C::kNumAcc + 1);
    auto cfull_bar = [&](int ew, int i) { return ebar0 + 8u * (ew * (C::kCSlots + C::kDSlots) + i); };
    auto dcfull_bar = [&](int ew, int j) { return ebar0 + 8u * (ew * (C::kCSlots + C::kDSlots) + C::kCSlots + j); };
    const uint32_t xfull_bar = bar0 + 8u * (2 * C::kStages + 2 * C::kNumAcc + 1 + C::kNumCBars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    int* sched = reinterpret_cast<int*>(smem + C::kOffSched);
    int* cnt = reinterpret_cast<int*>(smem + C::kOffCnt);

    // ---------------------------------------------------------------- prologue
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            // the A and the B producer each arrive (with their bytes) and the 32 scale-loader
            // lanes arrive once their copies have landed
            mbar_init(full_bar(s), 34);
            mbar_init(empty_bar(s), 1);    // tcgen05.commit of the MMA issuer
        }
        for (int b = 0; b < C::kNumAcc; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 4);   // one arrive per epilogue warp
        }
        mbar_init(mma_drain_bar, 1);
        for (int i = 0; i < C::kNumCBars; ++i) mbar_init(ebar0 + 8u * i, 1);   // TMA bytes of a C chunk
        mbar_init(xfull_bar, 4 * split);   // split-K: every epilogue warp of the cluster
        *abort_flag = 0;
        fence_mbar_init();
        if (p.K > 0) {          // a K-grouped call with K_total == 0 has no operand maps
            tma_prefetch_map(&tm_a);
            tma_prefetch_map(&tm_b);
        }
        tma_prefetch_map(&tm_d);
        if (p.has_c && !p.c_in_d) tma_prefetch_map(&tm_c);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    // the cluster's barriers are initialised before any CTA of it arrives on them remotely
    if (split > 1) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    // While the previous grid of the stream finishes (programmatic launch), a CTA that owns a
    // single dense tile asks L2 for that tile's B (the weights) with tensor-map prefetches
    // spread over four lanes.  A prefetch moves data from HBM into L2 only: nothing reaches
    // this SM before the dependency wait, and L2 is where every write of the previous grid
    // lands, so the loads after the wait see that grid's data whatever it wrote.
    if (p.prefetch_b && warp == 2 && lane < 4 && kind == kDense) {
        TileIter<BN> pit = tiles_of_cta<BN>(rank, split, kind);
        Tile ptl;
        if (pit.next(p, p.num_mb * p.num_nb, sched, cnt, ptl)) {
            for (int kb = lane; kb < ptl.nkb; kb += 4) {
                const int kc = (ptl.kb0 + kb) * 128;
                if constexpr (!kBmn) tma_prefetch_l2_2d(&tm_b, kc, ptl.b_coord);
                else
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h) tma_prefetch_l2_2d(&tm_b, ptl.n0 + h * 128, kc);
            }
        }
    }
    // Nothing above read global memory into the SM (the tensor maps are kernel parameters),
    // so the set-up overlaps the previous grid's tail under a programmatic launch; here its
    // results become visible.
    grid_dependency_wait();
    if (threadIdx.x == 0) grid_launch_dependents();
    // Group tables for the masked (tile prefix) and K-grouped (K-group prefix) layouts.
    int total_tiles = p.num_mb * p.num_nb;
    if (warp == 2) {
        if (kind == kMasked || kind == kKGrouped) {
            int run = 0;
            bool bad = false;
            for (int g0 = 0; g0 < p.G; g0 += 32) {
                const int g = g0 + lane;
                int v = 0;
                if (g < p.G) {
                    if (kind == kMasked) {
                        int mm = __ldg(p.masked_m + g);
                        if (mm < 0 || mm > p.M) bad = true;
                        mm = max(0, min(mm, p.M));
                        cnt[g] = mm;
                        v = ((mm + 127) / 128) * p.num_nb;
                    } else {
                        const int k = __ldg(p.ks + g);
                        if (k < 0 || (k & 127)) bad = true;
                        v = max(k, 0) / 128;
                    }
                }
                int incl = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                if (g < p.G) sched[g] = run + incl - v;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) sched[p.G] = run;
            bad = __any_sync(0xffffffffu, bad);
            if (lane == 0 && bad)
                record_status(p.status, kErrContract | (kind == kMasked ? kChkMaskRange : kChkKSegments));
            if (kind == kKGrouped && lane == 0 && (bad || run * 128 != p.K)) {
                if (!bad) record_status(p.status, kErrContract | kChkKSegments);
                sched[p.G] = -1;   // marks the whole call as invalid
            }
        }
    }
    if (kind == kMasked || kind == kKGrouped) __syncthreads();   // the group tables
    const uint32_t tmem_base = *tmem_slot;
    if (kind == kMasked) total_tiles = sched[p.G];
    if (kind == kKGrouped) total_tiles = sched[p.G] < 0 ? 0 : p.G * p.num_mb * p.num_nb;
    if (split > 1 && (p.kind != kDense || static_cast<int>(cluster_nctarank()) != split ||
                      static_cast<long long>(total_tiles) * split > gridDim.x)) {
        // the exchange assumes one tile per cluster of `split` CTAs: refuse anything else
        if (threadIdx.x == 0) record_status(p.status, kErrContract | kChkSplit);
        total_tiles = 0;
    }

    const WaitCtl wctl{abort_flag, p.status, p.timeout_ns};

    if (warp == 0 || warp == 8) {
        // ----------------------------------------------------- TMA producers of A
        // warp 0 fills the even stages of the global stage sequence, warp 8 the odd ones
        if (lane == 0) {
            const uint32_t par = warp == 0 ? 0u : 1u;
            int s = 0;
            uint32_t ph = 0, g = 0;
            bool stall = p.debug_stall != 0 && par == 0;
            uint32_t armed = 0, armed_par = 0;   // per-stage: armed at least once / parity
            bool aborted = false;
            TileIter<BN> it = tiles_of_cta<BN>(rank, split, kind);
            Tile tl;
            while (!aborted && it.next(p, total_tiles, sched, cnt, tl)) {
                for (int kb = 0; kb < tl.nkb; ++kb, ++g) {
                    if ((g & 1u) != par) {
                        if (++s == C::kStages) { s = 0; ph ^= 1u; }
                        continue;
                    }
                    if (!wait_bar(empty_bar(s), ph ^ 1u, wctl, kWaitProducer)) { aborted = true; break; }
                    if (stall) {
                        stall = false;   // leave this stage unarmed: the MMA issuer times out
                    } else {
                        const uint32_t fb = full_bar(s);
                        const uint32_t sa = sbase + C::kOffA + s * C::kABytes;
                        const int kc = (tl.kb0 + kb) * 128;
                        if constexpr (!kAmn) {
                            mbar_arrive_expect_tx(fb, p.a_box_rows * C::kBK);
                            tma_load_2d(sa, &tm_a, fb, kc, tl.a_coord);
                        } else {              // A [K][M]: one 128 (M) x 128 (K) box
                            mbar_arrive_expect_tx(fb, C::kABytes);
                            tma_load_2d(sa, &tm_a, fb, tl.a_coord, kc);
                        }
                        armed |= 1u << s;
                        armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    }
                    if (++s == C::kStages) { s = 0; ph ^= 1u; }
                }
            }
            if (aborted || *abort_flag) {
                // Bounded drain of loads that may still be landing in shared memory.
                for (int i = 0; i < C::kStages; ++i)
                    if (armed >> i & 1u) drain_bar(full_bar(i), armed_par >> i & 1u, 20000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdesc = make_idesc_mxf8(128, BN, kAmn, kBmn, kFp4B ? kFmtE2M1 : kFmtE4M3);
            // TMEM scale slots in rotation: FP4 B copies a scale word row at every K-group,
            // so it rotates over four slots (a slot is rewritten four K-groups after the MMAs
            // that read it were issued); FP8 scales change every fourth K-group, two slots.
            constexpr uint32_t kSfSlots = kFp4B ? 4u : 2u;
            static_assert(C::kSfCol0 + 16 * (kSfSlots - 1) + C::kSfCols <= 512, "TMEM columns of the scale slots");
            // Shared-memory descriptors of stage 0; a stage's descriptor adds its offset in
            // 16-byte units to the start-address field (shared addresses stay below 2^18, so
            // the 14-bit field never carries).  K step j of a stage: K-major operands advance
            // 32 bytes along the 128-byte swizzled rows, MN-major ones 4 KB (8 K rows of 128-wide
            // atoms 16 KB apart).
            const uint64_t a_desc0 = kAmn ? make_sdesc(sbase + C::kOffA, 16384, 1024, kLayoutSw128)
                                          : make_sdesc(sbase + C::kOffA, 0, 1024, kLayoutSw128);
            const uint64_t b_desc0 = kBmn ? make_sdesc(sbase + C::kOffB, 16384, 1024, kLayoutSw128)
                                          : make_sdesc(sbase + C::kOffB, 0, 1024, kLayoutSw128);
            constexpr uint32_t kAStep = kAmn ? 4096 / 16 : 32 / 16, kBStep = kBmn ? 4096 / 16 : 32 / 16;
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_ph = 0;
            uint32_t kcount = 0;    // scale-word copies issued (selects the TMEM scale slot)
            bool aborted = false;
            TileIter<BN> it = tiles_of_cta<BN>(rank, split, kind);
            Tile tl;
            // one stage: the scale words it carries (if it starts a packed word row) to TMEM,
            // its four MMAs, and the commit that frees it
            auto issue_stage = [&](int kb, uint32_t d_t) {
                const uint32_t sf_id = static_cast<uint32_t>(tl.kb0 + kb) & 3u;
                if (kFp4B || kb == 0 || sf_id == 0) {
                    // A packed word holds the scales of four consecutive K-groups: copy it at the
                    // tile's first K-group and at every fourth global K-group, alternating between
                    // two TMEM slots (the copy of the next word never overwrites one still read by
                    // MMAs in flight: tcgen05 operations of one thread execute in issue order).
                    ++kcount;
                    const uint32_t sfa_n = tmem_base + C::kSfCol0 + (kcount % kSfSlots) * 16;
                    const uint32_t ssfa = sbase + C::kOffSf + s * C::kSfSlotBytes;
                    fence_proxy_async_smem();    // scale words written by cp.async, read by tcgen05.cp
                    tc_cp_32x128b_warpx4(sfa_n, make_sdesc(ssfa, 0, 128, kLayoutNone));
#pragma unroll
                    for (int i = 0; i < C::kSfbAtoms; ++i)
                        tc_cp_32x128b_warpx4(sfa_n + 4 + 4 * i, make_sdesc(ssfa + C::kSfaBytes + 512 * i, 0, 128, kLayoutNone));
                }
                const uint32_t sfa_t = tmem_base + C::kSfCol0 + (kcount % kSfSlots) * 16;
                const uint32_t sfb_t = sfa_t + 4;
                const uint64_t ad = a_desc0 + static_cast<uint64_t>((s * C::kABytes) >> 4);
                const uint64_t bd = b_desc0 + static_cast<uint64_t>((s * C::kBBytes) >> 4);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // A: byte (K-group mod 4) of its word; FP4 B: byte j (the j-th 32-wide block
                    // of this K-group), otherwise the A choice
                    const uint32_t idesc = idesc_sf_ids(kIdesc, sf_id, kFp4B ? static_cast<uint32_t>(j) : sf_id);
                    tc_mma_mxf8(d_t, ad + kAStep * j, bd + kBStep * j, idesc, sfa_t, sfb_t, (kb | j) != 0);
                }
                tc_commit(empty_bar(s));
                if (++s == C::kStages) { s = 0; ph ^= 1u; }
            };
            while (!aborted && it.next(p, total_tiles, sched, cnt, tl)) {
                if (!wait_bar(acce_bar(acc), acc_ph ^ 1u, wctl, kWaitMma)) { aborted = true; break; }
                tc_fence_after();
                const uint32_t d_t = tmem_base + acc * BN;
                int kb = 0;
                while (kb < tl.nkb) {
                    // the next two stages: two non-blocking tests in flight together
                    const int s1 = s + 1 == C::kStages ? 0 : s + 1;
                    const uint32_t ph1 = s + 1 == C::kStages ? ph ^ 1u : ph;
                    const bool two = kb + 1 < tl.nkb;
                    const bool r0 = mbar_test_wait(full_bar(s), ph);
                    bool r1 = two && mbar_test_wait(full_bar(s1), ph1);
                    if (!r0) {
                        if (!wait_bar(full_bar(s), ph, wctl, kWaitMma)) { aborted = true; break; }
                        r1 = two && mbar_test_wait(full_bar(s1), ph1);
                    }
                    tc_fence_after();
                    issue_stage(kb++, d_t);
                    if (r1) issue_stage(kb++, d_t);
                }
                if (aborted) break;
                if (tl.nkb > 0) tc_commit(accf_bar(acc));
                else mbar_arrive(accf_bar(acc));
                if (++acc == C::kNumAcc) { acc = 0; acc_ph ^= 1u; }
            }
            // Wait (bounded) until every tensor-core operation issued here has finished.
            tc_commit(mma_drain_bar);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(mma_drain_bar, 0)) {
                if (globaltimer_ns() - t0 > p.timeout_ns) { record_status(p.status, kErrTimeout | kWaitDrain); break; }
            }
        }
        __syncwarp();
    } else if (warp == 2 || warp == 9) {
        // ----------------------------------------------------- TMA producers of B
        // warp 2 fills the even stages of the global stage sequence, warp 9 the odd ones
        if (lane == 0) {
            const uint32_t par = warp == 2 ? 0u : 1u;
            int s = 0;
            uint32_t ph = 0, g = 0;
            uint32_t armed = 0, armed_par = 0;   // stages whose B load this lane issued / parity
            bool aborted = false;
            TileIter<BN> it = tiles_of_cta<BN>(rank, split, kind);
            Tile tl;
            while (!aborted && it.next(p, total_tiles, sched, cnt, tl)) {
                for (int kb = 0; kb < tl.nkb; ++kb, ++g) {
                    if ((g & 1u) != par) {
                        if (++s == C::kStages) { s = 0; ph ^= 1u; }
                        continue;
                    }
                    if (!wait_bar(empty_bar(s), ph ^ 1u, wctl, kWaitProducerB)) { aborted = true; break; }
                    const uint32_t sb = sbase + C::kOffB + s * C::kBBytes;
                    const int kc = (tl.kb0 + kb) * 128;
                    {
                        const uint32_t fb = full_bar(s);
                        // packed FP4 B: the transaction counts the bytes read (two codes per
                        // byte), half the unpacked bytes the box fills in shared memory
                        mbar_arrive_expect_tx(fb, kFp4B ? C::kBBytes / 2 : C::kBBytes);
                        if constexpr (kSwiGLU) {
                            // B as [2G halves][I rows][K]: one box of the tile's 128 gate rows
                            // and the matching 128 up rows (half 2g, then 2g + 1)
                            tma_load_3d(sb, &tm_b, fb, kc, (tl.n0 / 256) * 128, 2 * tl.g);
                        } else if constexpr (!kBmn) {
                            tma_load_2d(sb, &tm_b, fb, kc, tl.b_coord);
                        } else {   // B [K][N] (grouped: [G*K][N]): 128 (N) x 128 (K) boxes
                            const int krow = static_cast<int>(tl.b_krow) + kc;
#pragma unroll
                            for (int h = 0; h < BN / 128; ++h)
                                tma_load_2d(sb + h * 16384, &tm_b, fb, tl.n0 + h * 128, krow);
                        }
                        armed |= 1u << s;
                        armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    }
                    if (++s == C::kStages) { s = 0; ph ^= 1u; }
                }
            }
            if (aborted || *abort_flag) {
                // Bounded drain of B loads that may still be landing in shared memory.
                for (int i = 0; i < C::kStages; ++i)
                    if (armed >> i & 1u) drain_bar(full_bar(i), armed_par >> i & 1u, 20000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 3) {
        // ----------------------------------------------------- scale loader
        // Walks every stage with the producers.  A stage that starts a packed word row (the
        // tile's first K-group and every fourth global K-group) receives the words of the
        // tile's 128 A rows and BN B rows by 4-byte cp.async, written straight into the 32x4
        // atom layout that tcgen05.cp reads (word (lane, j) of each atom holds MN index
        // j * 32 + lane; rows outside the problem are zero-filled).  Each lane's arrival on
        // every stage's full barrier fires when its copies have landed.
        int s = 0;
        uint32_t ph = 0;
        TileIter<BN> it = tiles_of_cta<BN>(rank, split, kind);
        Tile tl;
        bool aborted = false;
        while (!aborted && it.next(p, total_tiles, sched, cnt, tl, kind == kContiguous)) {
            const int32_t* pa0 = p.sfa + tl.sfa_g * p.sfa_gstride;
            const int32_t* pb0 = p.sfb + tl.g * p.sfb_gstride;
            for (int kb = 0; kb < tl.nkb; ++kb) {
                // warp-uniform decision: every lane leaves together on abort
                const bool ok = wait_bar(empty_bar(s), ph ^ 1u, wctl, kWaitScales);
                if (!__all_sync(0xffffffffu, ok)) { aborted = true; break; }
                if (kFp4B || kb == 0 || ((tl.kb0 + kb) & 3) == 0) {
                    const int kw = (tl.kb0 + kb) >> 2;
                    const int32_t* pa = pa0 + (long long)kw * p.sfa_ld;
                    const uint32_t da = sbase + C::kOffSf + s * C::kSfSlotBytes + lane * 16;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int row = tl.sfa_row + lane + 32 * j;
                        const bool in = row < p.sfa_rows;
                        cp_async_4(da + 4 * j, in ? pa + row : pa, in ? 4u : 0u);
                    }
                    // FP4 B: one word row per K-group (four 32-wide blocks); else per four
                    const int32_t* pb = pb0 + (long long)(kFp4B ? tl.kb0 + kb : kw) * p.sfb_ld;
                    const uint32_t db = da + C::kSfaBytes;
#pragma unroll
                    for (int i = 0; i < C::kSfbAtoms; ++i) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            int n = tl.n0 + i * 128 + j * 32 + lane;
                            if constexpr (kSwiGLU) n = swiglu_b_row(p, tl, i) - (tl.b_coord - tl.n0) + j * 32 + lane;
                            const bool in = n < p.N;
                            cp_async_4(db + i * 512 + 4 * j, in ? pb + (p.sfb_per_row ? n : (n >> 7)) : pb, in ? 4u : 0u);
                        }
                    }
                }
                cp_async_mbar_arrive(full_bar(s));
                if (++s == C::kStages) { s = 0; ph ^= 1u; }
            }
        }
        cp_async_wait_all();
        __syncwarp();
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM sub-partition this warp may read
        const int row = q * 32 + lane;          // tile row of this thread (= threadIdx.x - kEpiThread0)
        const bool f32 = p.d_f32 != 0;
        const int cw = f32 ? 32 : 64;           // columns per chunk: 128 bytes per row
        const bool kg = kind == kKGrouped;
        const int ew = warp - kEpiWarp0;        // epilogue warp index (slot region)
        const uint32_t cslot0 = sbase + C::kOffCSlots + ew * C::kCSlots * C::kSlotBytes;
        const uint8_t* cslot0_ptr = smem + C::kOffCSlots + ew * C::kCSlots * C::kSlotBytes;
        const uint32_t dslot0 = sbase + C::kOffDSlots + ew * C::kDSlots * C::kSlotBytes;
        uint8_t* dslot0_ptr = smem + C::kOffDSlots + ew * C::kDSlots * C::kSlotBytes;

        int acc = 0;
        uint32_t acc_ph = 0;
        bool aborted = false;
        TileIter<BN> it = tiles_of_cta<BN>(rank, split, kind);
        Tile tl;
        if constexpr (kSplit) {
            // split-K: one tile per cluster, exchanged through distributed shared memory
            uint32_t x_ph = 0;
            while (it.next(p, total_tiles, sched, cnt, tl)) {
                const SplitTile st{tl.valid_rows, tl.n0, p.N, tl.nkb, tl.d_row, p.has_c, p.d_f32, p.c, p.d};
                if (!split_k_tile<BN, C>(st, reinterpret_cast<float*>(smem + C::kOffA), tmem_base + acc * BN,
                                         accf_bar(acc), acc_ph, acce_bar(acc), xfull_bar, x_ph, wctl, rank, split)) {
                    aborted = true;
                    break;
                }
                x_ph ^= 1u;
                if (++acc == C::kNumAcc) { acc = 0; acc_ph ^= 1u; }
            }
        } else if constexpr (kSwiGLU) {
            // ------------------------------------------ SwiGLU + per-1x128 requantisation
            // Per tile and row: y[i] = SiLU(gate[i]) * up[i] for the tile's 128 outputs
            // (TMEM columns i and 128 + i), one UE8M0 scale for the row's 128 values, E4M3
            // codes into this warp's store slot (32 rows x 128 B, the TMA box) and a byte
            // store of the scale into its packed word.  One pass over TMEM keeps the row's 128
            // values in registers, so the single accumulator is free for the next tile's
            // MMAs before the codes are formed.
            const uint32_t qslot = dslot0;
            uint8_t* qslot_ptr = dslot0_ptr;
            while (it.next(p, total_tiles, sched, cnt, tl)) {
                const bool ok = wait_bar(accf_bar(acc), acc_ph, wctl, kWaitEpilogue);
                if (!__all_sync(0xffffffffu, ok)) { aborted = true; break; }
                tc_fence_after();
                const long long grow = tl.d_row + row;
                bool row_ok = row < tl.valid_rows;
                if (kind == kContiguous) {
                    const int mi = __ldg(p.m_indices + grow);
                    if (mi >= 0 && mi != tl.g) record_status(p.status, kErrContract | kChkMixedBlock);
                    row_ok = (mi == tl.g);
                }
                const int nb = tl.n0 / 256;                      // 128-wide output column block
                const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
                float y[128];
                float amax = 0.0f;
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 16) {
                    uint32_t g[16], u[16];
                    if (tl.nkb > 0) {
                        tmem_ld_32x32b_x16(tacc + c0, g);
                        tmem_ld_32x32b_x16(tacc + 128 + c0, u);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) g[i] = u[i] = 0u;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        y[c0 + i] = swiglu_value(g[i], u[i]);
                        amax = fmaxf(amax, fabsf(y[c0 + i]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce_bar(acc));        // the accumulator is free
                const int e = scale_exponent(amax);
                if (lane == 0) bulk_wait_group_read<0>();    // the slot's previous store has read it
                __syncwarp();
                uint8_t* rowp = qslot_ptr + lane * 128;
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t w[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        uint32_t word = 0;
#pragma unroll
                        for (int j = 0; j < 4; ++j) word |= e4m3(ldexpf(y[c0 + 4 * k + j], -e)) << (8 * j);
                        w[k] = word;
                    }
                    const int cell = (c0 / 32) * 2;               // 32 codes = two 16-byte cells
                    *reinterpret_cast<uint4*>(rowp + ((cell ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4*>(rowp + (((cell + 1) ^ (lane & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
                if (row_ok) {
                    const int sf_row = kind == kMasked ? tl.sfa_row + row : static_cast<int>(grow);
                    const int32_t* wp = p.sfq + (kind == kMasked ? tl.g * p.sfq_gstride : 0) +
                                        (long long)(nb >> 2) * p.sfq_ld + sf_row;
                    *(reinterpret_cast<uint8_t*>(const_cast<int32_t*>(wp)) + (nb & 3)) = static_cast<uint8_t>(e + 127);
                }
                // Dense rows past M are clipped by the TMA store; grouped layouts store only valid rows.
                if (kind == kDense || __all_sync(0xffffffffu, row_ok)) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_d, qslot, nb * 128, tl.d_y + q * 32);
                        bulk_commit_group();
                    }
                } else if (row_ok) {
                    uint8_t* dst = static_cast<uint8_t*>(p.d) + grow * (p.N / 2) + nb * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4*>(dst + 16 * j) = *reinterpret_cast<const uint4*>(rowp + ((j ^ (lane & 7)) << 4));
                }
                __syncwarp();
                if (++acc == C::kNumAcc) { acc = 0; acc_ph ^= 1u; }
            }
            if (lane == 0) bulk_wait_group_read<0>();
            __syncwarp();
        } else {
            // C prefetch cursor (lane 0): walks the same chunk sequence ahead, one 32-row x
            // 32-column FP32 chunk per C slot, each refilled as soon as it has been read.
            TileIter<BN> cit = tiles_of_cta<BN>(rank, split, kind);
            Tile ctl;
            bool c_have = false;
            int c_chunk = 0;
            uint32_t c_issued = 0;       // C chunks whose load has been issued
            auto issue_c = [&](uint32_t id) {
                const int sl = static_cast<int>(id % C::kCSlots);
                const uint32_t dst = cslot0 + sl * C::kSlotBytes;
                const uint32_t bar = cfull_bar(ew, sl);
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, C::kSlotBytes);
                const int x = ctl.n0 + c_chunk * 32;
                if (kg) tma_load_3d(dst, &tm_c, bar, x, ctl.d_y + q * 32, ctl.d_z);
                else tma_load_2d(dst, &tm_c, bar, x, ctl.d_y + q * 32);
                if (++c_chunk == (min(BN, p.N - ctl.n0) + 31) / 32) {
                    c_chunk = 0;
                    c_have = cit.next(p, total_tiles, sched, cnt, ctl);
                }
            };
            const bool load_c = p.has_c && !p.c_in_d;   // in place: the reduce-add brings C in
            if constexpr (C::kCSlots > 0) {
                if (lane == 0 && load_c) {
                    c_have = cit.next(p, total_tiles, sched, cnt, ctl);
                    while (c_have && c_issued < static_cast<uint32_t>(C::kCSlots)) issue_c(c_issued++);
                }
            }

            uint32_t chunk_id = 0;       // C chunks consumed so far
            uint32_t dchunk = 0;         // chunks stored through the store slots
            while (it.next(p, total_tiles, sched, cnt, tl)) {
                // the row's expert id is loaded before the accumulator wait (its latency
                // overlaps the wait instead of following it)
                const long long grow = tl.d_row + row;
                const int mi = kind == kContiguous ? __ldg(p.m_indices + grow) : 0;
                // warp-uniform decision before the .sync.aligned TMEM loads below
                const bool ok = wait_bar(accf_bar(acc), acc_ph, wctl, kWaitEpilogue);
                if (!__all_sync(0xffffffffu, ok)) { aborted = true; break; }
                tc_fence_after();
                bool row_ok = row < tl.valid_rows;
                if (kind == kContiguous) {
                    if (mi >= 0 && mi != tl.g) record_status(p.status, kErrContract | kChkMixedBlock);
                    row_ok = (mi == tl.g);
                }
                // Rows past the end of the D tensor are clipped by the TMA store; the masked and
                // contiguous layouts have rows inside D that must stay untouched.
                const bool use_tma = (kind == kDense || kg) || __all_sync(0xffffffffu, row_ok);
                const int ncols = min(BN, p.N - tl.n0);
                const int nch = (ncols + cw - 1) / cw;
                for (int ch = 0; ch < nch; ++ch) {
                    const int c0 = ch * cw;
                    uint32_t r[64];
                    if (tl.nkb > 0) {
                        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c0,
                                           *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                        if (!f32 && c0 + 32 < BN)
                            tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c0 + 32,
                                               *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 64; ++i) r[i] = 0u;
                    }
                    if (!f32 && !(c0 + 32 < BN)) {
#pragma unroll
                        for (int i = 32; i < 64; ++i) r[i] = 0u;
                    }
                    if (ch == nch - 1) {
                        // the accumulator buffer is free once its last columns are in registers
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acce_bar(acc));
                    }
                    // A 64-column BF16 chunk at the end of a BN = 224 tile would store into the
                    // neighbouring tile: such a chunk takes the per-thread path (no C in BF16).
                    if (use_tma && c0 + cw <= BN) {
                        const int dsl = static_cast<int>(dchunk % C::kDSlots);
                        const uint32_t d_addr = dslot0 + dsl * C::kSlotBytes;
                        uint8_t* drow = dslot0_ptr + dsl * C::kSlotBytes + lane * 128;
                        if (load_c) {       // FP32 chunks: add C
                            const uint8_t* crow;
                            if constexpr (C::kCSlots > 0) {
                                const int csl = static_cast<int>(chunk_id % C::kCSlots);
                                const bool okc = wait_bar(cfull_bar(ew, csl), (chunk_id / C::kCSlots) & 1u, wctl,
                                                          kWaitEpilogueC);
                                if (!__all_sync(0xffffffffu, okc)) { aborted = true; break; }
                                crow = cslot0_ptr + csl * C::kSlotBytes + lane * 128;
                            } else {
                                // no C slots (the widest tiles): this chunk's C lands in the store
                                // slot once the store issued from it has read it, and D replaces
                                // it in place
                                if (lane == 1) bulk_wait_group_read<0>();
                                __syncwarp();
                                const uint32_t bar = dcfull_bar(ew, dsl);
                                if (lane == 0) {
                                    fence_proxy_async_smem();
                                    mbar_arrive_expect_tx(bar, C::kSlotBytes);
                                    if (kg) tma_load_3d(d_addr, &tm_c, bar, tl.n0 + c0, tl.d_y + q * 32, tl.d_z);
                                    else tma_load_2d(d_addr, &tm_c, bar, tl.n0 + c0, tl.d_y + q * 32);
                                }
                                const bool okc = wait_bar(bar, (dchunk / C::kDSlots) & 1u, wctl, kWaitEpilogueC);
                                if (!__all_sync(0xffffffffu, okc)) { aborted = true; break; }
                                crow = drow;
                            }
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 cv = *reinterpret_cast<const float4*>(crow + ((j ^ (lane & 7)) << 4));
                                r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + cv.x);
                                r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + cv.y);
                                r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + cv.z);
                                r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + cv.w);
                            }
                            if constexpr (C::kCSlots > 0) {
                                // the C slot is read: refill it with the chunk kCSlots ahead
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0 && c_have) issue_c(c_issued++);
                                ++chunk_id;
                            }
                        }
                        // the store slot's previous store (kDSlots chunks ago) must have read it
                        if (lane == 1) {
                            if constexpr (C::kDSlots == 1) bulk_wait_group_read<0>();
                            else bulk_wait_group_read<C::kDSlots - 1>();
                        }
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            uint4* cell = reinterpret_cast<uint4*>(drow + ((j ^ (lane & 7)) << 4));
                            uint4 w;
                            if (f32) {
                                w = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                            } else {
                                uint32_t pk[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(
                                        __uint_as_float(r[8 * j + 2 * i]), __uint_as_float(r[8 * j + 2 * i + 1]));
                                    pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
                                }
                                w = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            }
                            *cell = w;
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 1) {
                            if (p.c_in_d) {
                                if (kg) tma_reduce_add_3d(&tm_d, d_addr, tl.n0 + c0, tl.d_y + q * 32, tl.d_z);
                                else tma_reduce_add_2d(&tm_d, d_addr, tl.n0 + c0, tl.d_y + q * 32);
                            } else {
                                if (kg) tma_store_3d(&tm_d, d_addr, tl.n0 + c0, tl.d_y + q * 32, tl.d_z);
                                else tma_store_2d(&tm_d, d_addr, tl.n0 + c0, tl.d_y + q * 32);
                            }
                            bulk_commit_group();
                        }
                        ++dchunk;
                    } else {
                        // Partially valid row group (no C in these layouts) or a chunk reaching past
                        // the tile: per-thread stores of the valid rows and columns.
                        if (row_ok) {
                            const int left = ncols - c0;
                            if (f32) {
                                float* dp = static_cast<float*>(p.d) + grow * p.N + tl.n0 + c0;
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    if (4 * j < left)
                                        *reinterpret_cast<uint4*>(dp + 4 * j) =
                                            make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                            } else {
                                __nv_bfloat16* dp = static_cast<__nv_bfloat16*>(p.d) + grow * p.N + tl.n0 + c0;
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    if (8 * j < left) {
                                        uint32_t pk[4];
#pragma unroll
                                        for (int i = 0; i < 4; ++i) {
                                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(
                                                __uint_as_float(r[8 * j + 2 * i]), __uint_as_float(r[8 * j + 2 * i + 1]));
                                            pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
                                        }
                                        *reinterpret_cast<uint4*>(dp + 8 * j) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                                    }
                                }
                            }
                        }
                    }
                }
                if (aborted) break;
                if (++acc == C::kNumAcc) { acc = 0; acc_ph ^= 1u; }
            }
            if constexpr (C::kCSlots > 0) {
                // C loads issued but never consumed (abort) must land before the CTA exits.
                if (lane == 0)
                    for (uint32_t c = chunk_id; c < c_issued; ++c)
                        drain_bar(cfull_bar(ew, static_cast<int>(c % C::kCSlots)), (c / C::kCSlots) & 1u, 20000000ull);
            }
            if (lane == 1) bulk_wait_group_read<0>();   // the slots are read; the stores complete with the grid
            __syncwarp();
        }   // not split-K
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    // split-K: peers read this CTA's exchange buffer until here
    if (split > 1) cluster_sync();
    else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace fg
