// fg_mqa.cu - FP8 MQA logits of the lightning indexer on tcgen05 tensor cores.
//
// "DeepGEMM Documentation", section 11 "Use V3.2 MQA Kernels for Indexers" (non-paged
// fp8_mqa_logits): for query token i and kv token j in [ks[i], ke[i])
//     out[i, j] = sum_h relu(q[i, h, :] . (kv[j, :] * sf[j])) * w[i, h]
// and -inf elsewhere when clean_logits is set.  Here H = 64 heads and D = 128.
//
// The contraction q[i, h, :] . kv[j, :] is an FP8 GEMM with kv tokens on the MMA's M
// axis (128 per tile) and (query token, head) on N: a tile is 128 kv tokens x 4 query
// tokens x 64 heads (N = 256), K = D = 128 (four K=32 MMAs of kind::f8f6f4: q and kv
// carry no block scales, the kv scale is applied in the epilogue).  With kv on M, each
// epilogue thread owns one kv token j (one TMEM lane) and finds all 64 heads of a query
// token in consecutive TMEM columns, so relu, the head weights and the head sum stay
// inside the thread; out[i, j..j+31] is then one coalesced store per warp.
//
// Warp roles (576 threads): warp 0 TMA (the group's q tile once per group of four query
// tokens, kv tiles through an 8-stage ring); warp 1 TMEM owner + MMA issuer; warps 2..17
// epilogue, one query token of the group per four warps (warp w reads TMEM lanes
// 32 (w mod 4) ..).
// Two 256-column accumulators alternate in TMEM.  Four tokens per tile halve the MMA
// issuer's per-tile work (waits, descriptors, commits) per logit, which bounded the
// two-token form.  Every wait is bounded (globaltimer); on expiry the CTA records a
// time-out in the status word and every role winds down.
#include <cuda_runtime.h>

#include "fg_gemm_kernel.cuh"
#include "fg_mqa.cuh"

namespace fg {
namespace {

constexpr int kHeads = 64, kDim = 128, kTok = kMqaTokens, kBN = kTok * kHeads;   // N = 256
constexpr int kStages = 8;
constexpr int kNumAcc = 2;                  // 256-column accumulators in TMEM
constexpr int kKvBytes = 128 * kDim;                                    // 16 KB kv tile
constexpr int kQBytes = kBN * kDim;                                     // 32 KB q tile
constexpr int kOffKv = 0;
constexpr int kOffQ = kOffKv + kStages * kKvBytes;                      // two q buffers
constexpr int kOffW = kOffQ + 2 * kQBytes;                              // per epilogue warp: its token's weights
constexpr int kEpiWarps = 4 * kTok;        // 4 TMEM lane quarters x 4 tokens
constexpr int kOffBar = kOffW + kEpiWarps * kHeads * 4;
constexpr int kNumBars = 2 * kStages + 2 + 2 + 2 * kNumAcc + 1;         // full, empty, qfull, qempty, accf, acce, drain
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
constexpr int kThreads = 64 + 32 * kEpiWarps;

// kv tiles [lo, hi) a group of query tokens touches; empty when hi <= lo.
__device__ __forceinline__ void group_range(const MqaParams& p, int i0, int& lo, int& hi) {
    int a = p.T, b = 0;
    for (int t = 0; t < kTok; ++t) {
        const int i = i0 + t;
        if (i >= p.S) break;
        const int s = max(__ldg(p.ks + i), 0), e = min(__ldg(p.ke + i), p.T);
        if (e > s) { a = min(a, s); b = max(b, e); }
    }
    lo = a / 128;
    hi = b > a ? (b + 127) / 128 : lo;
}

// Packed FP32 pairs for fma.rn.f32x2 (x in the low half).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Group visited by this CTA in round r: rounds deal the groups to the CTAs in snake order
// (CTA b takes slot b in even rounds and slot grid-1-b in odd ones), latest query tokens
// first.  Under causal ranges a group's cost grows with its tokens, so the costly groups
// go out first and alternate ends of the grid (max per-CTA tiles 127 -> 113 of a mean of
// 111 at S = T = 4096).  Returns -1 for an empty slot of the last round, kNoGroup past it.
constexpr int kNoGroup = -2;
__device__ __forceinline__ int group_of(int r, int groups) {
    const int c = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    if (r * c >= groups) return kNoGroup;
    const int slot = r * c + ((r & 1) ? c - 1 - b : b);
    return slot < groups ? groups - 1 - slot : -1;
}

__global__ void __launch_bounds__(kThreads, 1)
mqa_kernel(const MqaParams p, const __grid_constant__ MqaMaps maps) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = sbase + kOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto qfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
    auto qempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 4 + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 4 + kNumAcc + b); };
    const uint32_t drain_bar_addr = bar0 + 8u * (2 * kStages + 4 + 2 * kNumAcc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(qfull_bar(b), 1);
            mbar_init(qempty_bar(b), 1);
        }
        for (int b = 0; b < kNumAcc; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), kEpiWarps);   // one arrive per epilogue warp
        }
        mbar_init(drain_bar_addr, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&maps.q);
        tma_prefetch_map(&maps.kv);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    grid_dependency_wait();
    if (threadIdx.x == 0) grid_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtl wctl{abort_flag, p.status, p.timeout_ns};
    const int groups = (p.S + kTok - 1) / kTok;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producers
        if (lane == 0) {
            int qb = 0;
            uint32_t qph = 0;
            unsigned n = 0;                              // kv tile counter of this CTA
            uint32_t armed = 0, armed_par = 0;
            bool aborted = false;
            for (int r = 0, pr; !aborted && (pr = group_of(r, groups)) != kNoGroup; ++r) {
                if (pr < 0) continue;
                int lo, hi;
                group_range(p, pr * kTok, lo, hi);
                if (hi <= lo) continue;
                {
                    if (!wait_bar<false, false>(qempty_bar(qb), qph ^ 1u, wctl, kWaitProducer)) { aborted = true; break; }
                    mbar_arrive_expect_tx(qfull_bar(qb), kQBytes);
                    tma_load_2d(sbase + kOffQ + qb * kQBytes, &maps.q, qfull_bar(qb), 0, pr * kTok * kHeads);
                    if (++qb == 2) { qb = 0; qph ^= 1u; }
                }
                for (int t = lo; t < hi; ++t, ++n) {
                    const int s = static_cast<int>(n % kStages);
                    const uint32_t ph = (n / kStages) & 1u;
                    if (!wait_bar<false, false>(empty_bar(s), ph ^ 1u, wctl, kWaitProducer)) { aborted = true; break; }
                    mbar_arrive_expect_tx(full_bar(s), kKvBytes);
                    tma_load_2d(sbase + kOffKv + s * kKvBytes, &maps.kv, full_bar(s), 0, t * 128);
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                }
            }
            if (aborted || *abort_flag) {
                for (int i = 0; i < kStages; ++i)
                    if (armed >> i & 1u) drain_bar(full_bar(i), armed_par >> i & 1u, 20000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc_f8(128, kBN);
            int s = 0, qb = 0, acc = 0;
            uint32_t ph = 0, qph = 0, acc_ph = 0;
            bool aborted = false;
            for (int r = 0, pr; !aborted && (pr = group_of(r, groups)) != kNoGroup; ++r) {
                if (pr < 0) continue;
                int lo, hi;
                group_range(p, pr * kTok, lo, hi);
                if (hi <= lo) continue;
                if (!wait_bar<false, false>(qfull_bar(qb), qph, wctl, kWaitMma)) { aborted = true; break; }
                const uint32_t sq = sbase + kOffQ + qb * kQBytes;
                for (int t = lo; t < hi; ++t) {
                    if (!wait_bar<false, false>(acce_bar(acc), acc_ph ^ 1u, wctl, kWaitMma)) { aborted = true; break; }
                    if (!wait_bar<false, false>(full_bar(s), ph, wctl, kWaitMma)) { aborted = true; break; }
                    tc_fence_after();
                    const uint32_t skv = sbase + kOffKv + s * kKvBytes;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tc_mma_f8(tmem_base + acc * kBN, make_sdesc(skv + 32 * j, 0, 1024, kLayoutSw128),
                                  make_sdesc(sq + 32 * j, 0, 1024, kLayoutSw128), idesc, j != 0);
                    tc_commit(empty_bar(s));
                    tc_commit(accf_bar(acc));
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                    if (++acc == kNumAcc) { acc = 0; acc_ph ^= 1u; }
                }
                if (aborted) break;
                tc_commit(qempty_bar(qb));      // the group's q tile is free once its MMAs are done
                if (++qb == 2) { qb = 0; qph ^= 1u; }
            }
            // bounded wait until every tensor-core operation issued here has finished
            tc_commit(drain_bar_addr);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain_bar_addr, 0)) {
                if (globaltimer_ns() - t0 > p.timeout_ns) { record_status(p.status, kErrTimeout | kWaitDrain); break; }
            }
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------------- epilogue (warps 2..17)
        const int q = warp & 3;                       // TMEM lanes 32q..32q+31
        const int row = q * 32 + lane;
        const int e = warp - 2;
        const int tok = e >> 2;                       // the group's query token this warp reduces
        const int et = static_cast<int>(threadIdx.x) - 64;   // 0..511 over the epilogue warps
        // each epilogue warp keeps its own copy of its token's head weights (no cross-warp barrier)
        float* w_s = reinterpret_cast<float*>(smem + kOffW) + e * kHeads;
        int acc = 0;
        uint32_t acc_ph = 0;
        bool aborted = false;
        for (int r = 0, pr; !aborted && (pr = group_of(r, groups)) != kNoGroup; ++r) {
            if (pr < 0) continue;
            const int i0 = pr * kTok;
            const int i = i0 + tok;
            int lo, hi;
            group_range(p, i0, lo, hi);
            __syncwarp();
#pragma unroll
            for (int c = 0; c < kHeads / 32; ++c)
                w_s[c * 32 + lane] = i < p.S ? __ldg(p.weights + (long long)i * kHeads + c * 32 + lane) : 0.0f;
            __syncwarp();
            const int ks_i = i < p.S ? max(__ldg(p.ks + i), 0) : 0;
            const int ke_i = i < p.S ? min(__ldg(p.ke + i), p.T) : 0;
            if (p.clean) {
                // -inf outside the kv tiles this group visits
                const int c0 = hi > lo ? lo * 128 : p.T, c1 = hi > lo ? min(hi * 128, p.T) : p.T;
                for (int t = 0; t < kTok; ++t) {
                    const int it = i0 + t;
                    if (it >= p.S) break;
                    float* orow = p.out + (long long)it * p.T;
                    for (int j = et; j < c0; j += 32 * kEpiWarps) orow[j] = -__int_as_float(0x7f800000);
                    for (int j = c1 + et; j < p.T; j += 32 * kEpiWarps) orow[j] = -__int_as_float(0x7f800000);
                }
            }
            const float4* w4 = reinterpret_cast<const float4*>(w_s);
            // kv scales are read one tile ahead: a global load right before the math would
            // put its latency on every tile
            float sf_next = (lo < hi && lo * 128 + row < p.T) ? __ldg(p.kv_sf + lo * 128 + row) : 0.0f;
            for (int tile = lo; tile < hi; ++tile) {
                const int j = tile * 128 + row;
                const float sfj = sf_next;
                const int jn = j + 128;
                sf_next = (tile + 1 < hi && jn < p.T) ? __ldg(p.kv_sf + jn) : 0.0f;
                const bool ok = wait_bar<false, false>(accf_bar(acc), acc_ph, wctl, kWaitEpilogue);
                if (!__all_sync(0xffffffffu, ok)) { aborted = true; break; }
                tc_fence_after();
                const uint32_t ta = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN + tok * kHeads;
                // eight independent partial sums: the head sum is FMA-latency bound as one chain.
                // For sf[j] > 0, relu(x * sf) = sf * relu(x): the scale is applied once after
                // the sum; any other scale takes the literal per-head form.  The 64 heads come
                // from TMEM in two halves of 32 registers (the block's register budget).
                // Partial sums in packed pairs: fma.rn.f32x2 does two of the head products per
                // instruction (same rounding and the same partial-sum assignment as scalar FMAs).
                uint64_t part2[4] = {0ull, 0ull, 0ull, 0ull};
                const bool pos = sfj > 0.0f;
                const ulonglong2* w2 = reinterpret_cast<const ulonglong2*>(w4);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(ta + 32 * hh, v);
                    tmem_wait_ld();
                    if (hh == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acce_bar(acc));    // this warp's part is in registers
                    }
                    if (pos) {
#pragma unroll
                        for (int h4 = 0; h4 < 8; ++h4) {
                            const ulonglong2 wv = w2[hh * 8 + h4];
                            uint64_t* pc = part2 + 2 * (h4 & 1);
                            float r[4];
#pragma unroll
                            for (int c = 0; c < 4; ++c) r[c] = fmaxf(__uint_as_float(v[4 * h4 + c]), 0.0f);
                            pc[0] = ffma2(pack_f32x2(r[0], r[1]), wv.x, pc[0]);
                            pc[1] = ffma2(pack_f32x2(r[2], r[3]), wv.y, pc[1]);
                        }
                    } else {
#pragma unroll
                        for (int h4 = 0; h4 < 8; ++h4) {
                            const ulonglong2 wv = w2[hh * 8 + h4];
                            uint64_t* pc = part2 + 2 * (h4 & 1);
                            float r[4];
#pragma unroll
                            for (int c = 0; c < 4; ++c) r[c] = fmaxf(__uint_as_float(v[4 * h4 + c]) * sfj, 0.0f);
                            pc[0] = ffma2(pack_f32x2(r[0], r[1]), wv.x, pc[0]);
                            pc[1] = ffma2(pack_f32x2(r[2], r[3]), wv.y, pc[1]);
                        }
                    }
                }
                float part[8];
#pragma unroll
                for (int c = 0; c < 4; ++c) unpack_f32x2(part2[c], part[2 * c], part[2 * c + 1]);
                const float sum = (((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]))) *
                                  (pos ? sfj : 1.0f);
                if (i < p.S && j < p.T) {
                    if (j >= ks_i && j < ke_i) p.out[(long long)i * p.T + j] = sum;
                    else if (p.clean) p.out[(long long)i * p.T + j] = -__int_as_float(0x7f800000);
                }
                if (++acc == kNumAcc) { acc = 0; acc_ph ^= 1u; }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace

cudaError_t launch_mqa(const MqaParams& p, const MqaMaps& maps, int grid, cudaStream_t stream) {
    static bool configured[256] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        err = cudaFuncSetAttribute(mqa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (err != cudaSuccess) return err;
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, mqa_kernel, p, maps);
}

}  // namespace fg
