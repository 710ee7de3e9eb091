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
// CUDA-core FMA pass).
//
// Warp roles (224 threads):
//   warp 0      TMA producer: A and B tiles into a ring of shared-memory stages
//   warp 1      TMEM owner + MMA issuer (one elected lane)
//   warp 2      scale loader: packed UE8M0 words into the tcgen05.cp layout
//   warps 3..6  epilogue: TMEM -> registers (+C) -> BF16/FP32 -> global memory
// Every role walks the same static persistent tile sequence (tile = blockIdx.x +
// i * gridDim.x), decoded from device-resident segment data without host sync.
//
// Every wait is bounded (globaltimer); on expiry the CTA records a time-out in the
// device status word, raises a shared abort flag that every other wait observes,
// drains its own in-flight tensor-core work and TMA loads (again bounded), frees TMEM
// and returns.  Nothing traps.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "fg_ptx.cuh"

namespace fg {

enum GemmKind : int { kDense = 0, kContiguous = 1, kMasked = 2, kKGrouped = 3 };

// Device status codes (the word keeps the first event).
enum : int {
    kErrContract = 0x100,      // | check id
    kErrTimeout = 0x200,       // | where
    kChkGroupIndex = 1,        // m_indices names a group >= G
    kChkMixedBlock = 2,        // a row names another group than its block
    kChkMaskRange = 3,         // masked_m outside [0, M_max]
    kChkKSegments = 4,         // ks not multiples of 128 / negative / wrong sum
    kWaitProducer = 1, kWaitMma = 2, kWaitScales = 3, kWaitEpilogue = 4, kWaitDrain = 5,
};

constexpr int kMaxGroups = 1024;  // masked / K-grouped groups held in shared memory

struct GemmParams {
    int kind;
    int M, N, K;           // dense M,N,K | contiguous M_total | masked M_max | K-grouped M,N,K_total
    int G;
    int d_f32, has_c;
    int num_mb, num_nb;    // tile grid of one group
    const int32_t* sfa;
    const int32_t* sfb;
    int sfa_ld, sfb_ld;    // int32 words per packed-word row of the scale arrays
    long long sfa_gstride, sfb_gstride;  // words between groups (masked SFA, grouped SFB)
    int sfa_rows;          // MN extent of the SFA rows
    const int32_t* m_indices;
    const int32_t* masked_m;
    const int32_t* ks;
    const float* c;
    void* d;
    int* status;
    unsigned long long timeout_ns;
    int debug_stall;
};

template <int BN>
struct TileCfg {
    static constexpr int kBM = 128, kBK = 128;
    static constexpr int kSfbAtoms = (BN + 127) / 128;
    static constexpr int kSfCols = 4 + 4 * kSfbAtoms;   // TMEM columns of one scale slot
    static constexpr int kNumAcc = (2 * BN + 2 * kSfCols <= 512) ? 2 : 1;
    static constexpr int kSfCol0 = kNumAcc * BN;
    static constexpr int kABytes = kBM * kBK;             // 16 KB
    static constexpr int kBBytes = BN * kBK;
    static constexpr int kSfaBytes = 512;
    static constexpr int kSfbBytes = kSfbAtoms * 512;
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static constexpr int kStages0 = (200 * 1024) / kStageBytes;
    static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kABytes;
    static constexpr int kOffSfa = kOffB + kStages * kBBytes;
    static constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
    static constexpr int kOffBar = kOffSfb + kStages * kSfbBytes;
    static constexpr int kNumBars = 2 * kStages + 2 * kNumAcc + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;        // tmem addr, abort flag
    static constexpr int kOffSched = kOffMisc + 16;                // int[kMaxGroups + 1]
    static constexpr int kOffCnt = kOffSched + (kMaxGroups + 1) * 4;
    static constexpr int kSmemBytes = kOffCnt + kMaxGroups * 4 + 1024;  // + alignment slack
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

struct Tile {
    int g, n0;
    int a_coord, b_coord;   // NT: rows in the A/B maps; TN: columns (m0 / n0)
    int kb0, nkb;           // first global K-group and number of K-groups
    int valid_rows;         // rows [0, valid_rows) of the tile lie inside the problem
    long long d_row;        // row of D (and C) that holds the tile's row 0
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
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtl& w, int where) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*w.abort) return false;
        if (globaltimer_ns() - t0 > w.timeout_ns) {
            *w.abort = 1;
            record_status(w.status, kErrTimeout | where);
            return false;
        }
    }
}

template <int BN>
__device__ __forceinline__ Tile decode_tile(const GemmParams& p, int t, const int* sched,
                                            const int* cnt, int& cursor) {
    Tile tl;
    tl.skip = false;
    tl.g = 0;
    tl.kb0 = 0;
    tl.nkb = p.K / 128;
    tl.sfa_g = 0;
    if (p.kind == kDense) {
        const int mb = t % p.num_mb, nb = t / p.num_mb;
        tl.n0 = nb * BN;
        tl.a_coord = mb * 128;
        tl.b_coord = tl.n0;
        tl.valid_rows = min(128, p.M - mb * 128);
        tl.d_row = mb * 128;
        tl.sfa_row = mb * 128;
    } else if (p.kind == kContiguous) {
        const int mb = t / p.num_nb, nb = t % p.num_nb;
        const int g = __ldg(p.m_indices + (long long)mb * 128);
        tl.n0 = nb * BN;
        if (g < 0 || g >= p.G) {
            if (g >= p.G) record_status(p.status, kErrContract | kChkGroupIndex);
            tl.skip = true;
        }
        tl.g = g < 0 ? 0 : (g >= p.G ? 0 : g);
        tl.a_coord = mb * 128;
        tl.b_coord = tl.g * p.N + tl.n0;
        tl.valid_rows = 128;
        tl.d_row = (long long)mb * 128;
        tl.sfa_row = mb * 128;
    } else if (p.kind == kMasked) {
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
        tl.sfa_row = mb * 128;
    }
    return tl;
}

template <int BN, bool kTN>
__global__ void __launch_bounds__(224, 1)
fg_gemm_kernel(const GemmParams p, const __grid_constant__ CUtensorMap tm_a,
               const __grid_constant__ CUtensorMap tm_b) {
    using C = TileCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t bar0 = sbase + C::kOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * C::kStages + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * C::kStages + C::kNumAcc + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * C::kStages + 2 * C::kNumAcc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    int* sched = reinterpret_cast<int*>(smem + C::kOffSched);
    int* cnt = reinterpret_cast<int*>(smem + C::kOffCnt);

    // ---------------------------------------------------------------- prologue
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(full_bar(s), 2);     // producer arrive (+ TMA bytes) and scale loader
            mbar_init(empty_bar(s), 1);    // tcgen05.commit of the MMA issuer
        }
        for (int b = 0; b < C::kNumAcc; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 4);     // one arrive per epilogue warp
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (p.K > 0) {          // a K-grouped call with K_total == 0 has no operand maps
            tma_prefetch_map(&tm_a);
            tma_prefetch_map(&tm_b);
        }
    }
    // Group tables for the masked (tile prefix) and K-grouped (K-group prefix) layouts.
    int total_tiles = p.num_mb * p.num_nb;
    if (warp == 2) {
        if (p.kind == kMasked || p.kind == kKGrouped) {
            int run = 0;
            bool bad = false;
            for (int g0 = 0; g0 < p.G; g0 += 32) {
                const int g = g0 + lane;
                int v = 0;
                if (g < p.G) {
                    if (p.kind == kMasked) {
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
                record_status(p.status, kErrContract | (p.kind == kMasked ? kChkMaskRange : kChkKSegments));
            if (p.kind == kKGrouped && lane == 0 && (bad || run * 128 != p.K)) {
                if (!bad) record_status(p.status, kErrContract | kChkKSegments);
                sched[p.G] = -1;   // marks the whole call as invalid
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    bool invalid = false;
    if (p.kind == kMasked) total_tiles = sched[p.G];
    if (p.kind == kKGrouped) {
        invalid = sched[p.G] < 0;
        total_tiles = p.G * p.num_mb * p.num_nb;
    }
    if (invalid) total_tiles = 0;

    const WaitCtl wctl{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int cursor = 0;
            bool stall = p.debug_stall != 0;
            uint32_t armed = 0, armed_par = 0;   // per-stage: armed at least once / parity
            bool aborted = false;
            for (int t = blockIdx.x; t < total_tiles && !aborted; t += gridDim.x) {
                const Tile tl = decode_tile<BN>(p, t, sched, cnt, cursor);
                if (tl.skip) continue;
                for (int kb = 0; kb < tl.nkb; ++kb) {
                    if (!wait_bar(empty_bar(s), ph ^ 1u, wctl, kWaitProducer)) { aborted = true; break; }
                    if (stall) {
                        stall = false;   // leave this stage unarmed: the MMA issuer times out
                    } else {
                        const uint32_t fb = full_bar(s);
                        mbar_arrive_expect_tx(fb, C::kABytes + C::kBBytes);
                        const uint32_t sa = sbase + C::kOffA + s * C::kABytes;
                        const uint32_t sb = sbase + C::kOffB + s * C::kBBytes;
                        const int kc = (tl.kb0 + kb) * 128;
                        if (!kTN) {
                            tma_load_2d(sa, &tm_a, fb, kc, tl.a_coord);
                            tma_load_2d(sb, &tm_b, fb, kc, tl.b_coord);
                        } else {
                            tma_load_2d(sa, &tm_a, fb, tl.a_coord, kc);
#pragma unroll
                            for (int h = 0; h < BN / 128; ++h)
                                tma_load_2d(sb + h * 16384, &tm_b, fb, tl.b_coord + h * 128, kc);
                        }
                        armed |= 1u << s;
                        armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    }
                    if (++s == C::kStages) { s = 0; ph ^= 1u; }
                }
            }
            if (aborted || *abort_flag) {
                // Bounded drain of loads that may still be landing in shared memory.
                WaitCtl quick{abort_flag, p.status, 20000000ull};
                int dummy = 0;
                for (int i = 0; i < C::kStages; ++i) {
                    if (!(armed >> i & 1u)) continue;
                    const uint32_t par = armed_par >> i & 1u;
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(full_bar(i), par) && globaltimer_ns() - t0 < quick.timeout_ns) ++dummy;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdesc = make_idesc_mxf8(128, BN, kTN, kTN);
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_ph = 0;
            int cursor = 0;
            uint32_t kcount = 0;
            bool aborted = false;
            for (int t = blockIdx.x; t < total_tiles && !aborted; t += gridDim.x) {
                const Tile tl = decode_tile<BN>(p, t, sched, cnt, cursor);
                if (tl.skip) continue;
                if (!wait_bar(acce_bar(acc), acc_ph ^ 1u, wctl, kWaitMma)) { aborted = true; break; }
                tc_fence_after();
                const uint32_t d_t = tmem_base + acc * BN;
                for (int kb = 0; kb < tl.nkb; ++kb) {
                    if (!wait_bar(full_bar(s), ph, wctl, kWaitMma)) { aborted = true; break; }
                    tc_fence_after();
                    const uint32_t slot = kcount & 1u;
                    const uint32_t sfa_t = tmem_base + C::kSfCol0 + slot * C::kSfCols;
                    const uint32_t sfb_t = sfa_t + 4;
                    const uint32_t ssfa = sbase + C::kOffSfa + s * C::kSfaBytes;
                    const uint32_t ssfb = sbase + C::kOffSfb + s * C::kSfbBytes;
                    tc_cp_32x128b_warpx4(sfa_t, make_sdesc(ssfa, 0, 128, kLayoutNone));
#pragma unroll
                    for (int i = 0; i < C::kSfbAtoms; ++i)
                        tc_cp_32x128b_warpx4(sfb_t + 4 * i, make_sdesc(ssfb + 512 * i, 0, 128, kLayoutNone));
                    const uint32_t sf_id = static_cast<uint32_t>(tl.kb0 + kb) & 3u;
                    const uint32_t idesc = idesc_sf_ids(kIdesc, sf_id, sf_id);
                    const uint32_t sa = sbase + C::kOffA + s * C::kABytes;
                    const uint32_t sb = sbase + C::kOffB + s * C::kBBytes;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint64_t ad, bd;
                        if (!kTN) {   // K-major, 128-byte rows, 8-row swizzle atoms 1024 B apart
                            ad = make_sdesc(sa + 32 * j, 0, 1024, kLayoutSw128);
                            bd = make_sdesc(sb + 32 * j, 0, 1024, kLayoutSw128);
                        } else {      // MN-major: 128-byte MN atoms 16 KB apart, 8 K rows per 1024 B
                            ad = make_sdesc(sa + 4096 * j, 16384, 1024, kLayoutSw128);
                            bd = make_sdesc(sb + 4096 * j, 16384, 1024, kLayoutSw128);
                        }
                        tc_mma_mxf8(d_t, ad, bd, idesc, sfa_t, sfb_t, (kb | j) != 0);
                    }
                    tc_commit(empty_bar(s));
                    ++kcount;
                    if (++s == C::kStages) { s = 0; ph ^= 1u; }
                }
                if (aborted) break;
                if (tl.nkb > 0) tc_commit(accf_bar(acc)); else mbar_arrive(accf_bar(acc));
                if (++acc == C::kNumAcc) { acc = 0; acc_ph ^= 1u; }
            }
            // Wait (bounded) until every tensor-core operation issued here has finished.
            tc_commit(drain_bar);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain_bar, 0)) {
                if (globaltimer_ns() - t0 > p.timeout_ns) { record_status(p.status, kErrTimeout | kWaitDrain); break; }
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ----------------------------------------------------- scale loader
        int s = 0;
        uint32_t ph = 0;
        int cursor = 0;
        bool aborted = false;
        for (int t = blockIdx.x; t < total_tiles && !aborted; t += gridDim.x) {
            const Tile tl = decode_tile<BN>(p, t, sched, cnt, cursor);
            if (tl.skip) continue;
            for (int kb = 0; kb < tl.nkb; ++kb) {
                // warp-uniform decision: every lane leaves together on abort
                const bool ok = wait_bar(empty_bar(s), ph ^ 1u, wctl, kWaitScales);
                if (!__all_sync(0xffffffffu, ok)) { aborted = true; break; }
                const int kw = (tl.kb0 + kb) >> 2;
                const int32_t* pa = p.sfa + tl.sfa_g * p.sfa_gstride + (long long)kw * p.sfa_ld;
                int4 va;
                {
                    int v[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int row = tl.sfa_row + lane + 32 * j;
                        v[j] = row < p.sfa_rows ? __ldg(pa + row) : 0;
                    }
                    va = make_int4(v[0], v[1], v[2], v[3]);
                }
                // word (lane, j) of the 32x4 atom holds MN index j * 32 + lane
                *reinterpret_cast<int4*>(smem + C::kOffSfa + s * C::kSfaBytes + lane * 16) = va;
                const int32_t* pb = p.sfb + tl.g * p.sfb_gstride + (long long)kw * p.sfb_ld;
#pragma unroll
                for (int i = 0; i < C::kSfbAtoms; ++i) {
                    int v[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int n = tl.n0 + i * 128 + j * 32 + lane;
                        v[j] = n < p.N ? __ldg(pb + (kTN ? n : (n >> 7))) : 0;
                    }
                    *reinterpret_cast<int4*>(smem + C::kOffSfb + s * C::kSfbBytes + i * 512 + lane * 16) =
                        make_int4(v[0], v[1], v[2], v[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_bar(s));
                if (++s == C::kStages) { s = 0; ph ^= 1u; }
            }
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM sub-partition this warp may read
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t acc_ph = 0;
        int cursor = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
            const Tile tl = decode_tile<BN>(p, t, sched, cnt, cursor);
            if (tl.skip) continue;
            // warp-uniform decision before the .sync.aligned TMEM loads below
            const bool ok = wait_bar(accf_bar(acc), acc_ph, wctl, kWaitEpilogue);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const long long grow = tl.d_row + row;
            bool row_ok = row < tl.valid_rows;
            if (p.kind == kContiguous) {
                const int mi = __ldg(p.m_indices + grow);
                if (mi >= 0 && mi != tl.g) record_status(p.status, kErrContract | kChkMixedBlock);
                row_ok = (mi == tl.g);
            }
            for (int c0 = 0; c0 < BN; c0 += 32) {
                const int n = tl.n0 + c0;
                if (n >= p.N) break;
                uint32_t r[32];
                if (tl.nkb > 0) {
                    tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c0, r);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = 0u;
                }
                if (!row_ok) continue;
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                const int halves = (p.N - n) >= 32 ? 2 : 1;
                if (p.has_c) {
                    const float* cp = p.c + grow * p.N + n;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h < halves) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float4 cv = *reinterpret_cast<const float4*>(cp + h * 16 + i * 4);
                                v[h * 16 + i * 4 + 0] += cv.x;
                                v[h * 16 + i * 4 + 1] += cv.y;
                                v[h * 16 + i * 4 + 2] += cv.z;
                                v[h * 16 + i * 4 + 3] += cv.w;
                            }
                        }
                    }
                }
                if (p.d_f32) {
                    float* dp = static_cast<float*>(p.d) + grow * p.N + n;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h < halves) {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                *reinterpret_cast<float4*>(dp + h * 16 + i * 4) =
                                    make_float4(v[h * 16 + i * 4], v[h * 16 + i * 4 + 1],
                                                v[h * 16 + i * 4 + 2], v[h * 16 + i * 4 + 3]);
                        }
                    }
                } else {
                    __nv_bfloat16* dp = static_cast<__nv_bfloat16*>(p.d) + grow * p.N + n;
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                        w[i] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h < halves) {
#pragma unroll
                            for (int i = 0; i < 2; ++i)
                                *reinterpret_cast<uint4*>(dp + h * 16 + i * 8) =
                                    make_uint4(w[h * 8 + i * 4], w[h * 8 + i * 4 + 1],
                                               w[h * 8 + i * 4 + 2], w[h * 8 + i * 4 + 3]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(acc));
            if (++acc == C::kNumAcc) { acc = 0; acc_ph ^= 1u; }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace fg
