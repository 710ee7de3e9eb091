/*
 * fg.h - C ABI of the fine-grained-scaled FP8 (E4M3) GEMM library for sm_103a.
 *
 * What the library computes is stated on the DeepGEMM pages:
 *   - "DeepGEMM Documentation" (docsearch index), section 4 "Understand DeepGEMM GEMM
 *     Naming and Layouts": D = C + A @ B; NT means non-transposed A, transposed B, so
 *     fp8_gemm_nt computes D = C + A @ B.T; SM100 scaling factors are packed UE8M0,
 *     four per 32-bit integer, and the LHS scaling factors are TMA-aligned and
 *     transposed (MN-major).
 *   - same page, section 9 "Use Normal and Grouped GEMM Kernels", and the
 *     yuguo-Jack/DeepGEMM README, "Interfaces > Notices", "Grouped GEMMs (contiguous
 *     layout)" and "Grouped GEMMs (masked layout)": the M-grouped contiguous, the
 *     M-grouped masked and the K-grouped (weight-gradient, TN) variants.
 *   - same page, section 10 "Use DeepGEMM Utility Functions": set/get_num_sms,
 *     get_mk_alignment_for_contiguous_layout, get_tma_aligned_size.
 *
 * Conventions shared by every GEMM entry point
 *   - All array arguments are DEVICE pointers owned by the caller; the library never
 *     frees, keeps or allocates them, and allocates nothing per call.
 *   - FP8 operands are E4M3 bytes (OCP "fn": bias 7, no inf, S.1111.111 = NaN).
 *   - Scale factors are UE8M0 (value 2^(u-127)), packed four per int32: byte j
 *     (bits 8j..8j+7) of word w is the scale of K-group 4w+j, a K-group being 128
 *     consecutive K elements.  Packed scale arrays are MN-major:
 *     [ceil(K/512)][align4(MN)] int32, with align4(x) = x rounded up to a multiple
 *     of 4 (16 bytes).  Padding entries are ignored.
 *   - A scales are one per row per K-group (1x128).  B scales of the NT calls are
 *     one per 128x128 block (MN index = n / 128); the K-grouped call takes 1x128
 *     scales along K for both operands; the FP8 x FP4 calls (below) take packed E2M1 B
 *     with one scale per 32 K elements of a row.
 *   - C is optional FP32 and is accepted only with an FP32 D.  D may alias C (the same
 *     pointer: in-place accumulation, D += A @ B^T; the kernels then read no C of their own
 *     and add the product onto D with TMA reduce-adds, one FP32 add per element performed
 *     in L2).  C and D that overlap without being the same array are not supported.
 *     A BF16 D is round-to-nearest-even of the FP32 accumulator.
 *   - Alignment: A, B, C, D and the scale arrays must be 16-byte aligned;
 *     index arrays 4-byte aligned.  K (or every K segment) is a multiple of 128,
 *     N a multiple of 16.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; 0 is the legacy default
 *     stream): no host synchronisation, no allocation.  The current CUDA device must
 *     own all pointers.
 *   - Return value: FG_OK, or a negative fg_status.  Host-side argument errors return
 *     FG_ERR_INVALID_ARG / FG_ERR_UNSUPPORTED before anything is launched.  A launch
 *     failure returns FG_ERR_CUDA.  Contract violations found on the device (index or
 *     mask out of range, bad K segments) and internal wait time-outs never trap: the
 *     kernel skips the offending tile (or the whole call), records the first such
 *     event in a per-device status word and returns; fg_get_device_error reads it.
 *   - Results are deterministic: every element of D is written once by one tile (with D
 *     aliasing C, added onto once by one TMA reduce-add); when a dense GEMM with few
 *     tiles is split along K, the partial tiles are summed in a fixed order.
 *   - Environment switches (tuning and diagnosis aids; the defaults are the measured
 *     best): FG_FORCE_BN=64|128|192|224|256 forces the N tile where that width applies;
 *     FG_FORCE_SPLIT=1|2|4|8 forces the dense split-K cluster size (a split that cannot
 *     run falls back to the cost model); FG_PREFETCH_B=0 turns off the L2 prefetch of a
 *     single-tile CTA's B before its grid-dependency wait; FG_PRINT_CONFIGS=1 prints each
 *     launch's tiling to stderr.  Only a split changes the FP32 summation order; every
 *     choice stays within the stated tolerance.
 */
#ifndef FG_H
#define FG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, so a cudaStream_t (or torch's stream handle) passes as is. */
typedef struct CUstream_st* fg_stream_t;

typedef enum {
    FG_OK = 0,
    FG_ERR_INVALID_ARG = -1,       /* null/misaligned pointer, bad shape or dtype code */
    FG_ERR_UNSUPPORTED = -2,       /* valid but not provided (e.g. C with a BF16 D)    */
    FG_ERR_CUDA = -3,              /* a CUDA runtime/driver call failed (no device...)  */
    FG_ERR_DEVICE_CONTRACT = -4,   /* device-side index/mask/segment contract violated  */
    FG_ERR_DEVICE_TIMEOUT = -5     /* a bounded wait inside a kernel ran out            */
} fg_status;

typedef enum { FG_BF16 = 0, FG_F32 = 1 } fg_dtype;

/*
 * Dense NT GEMM:  D[M,N] = C[M,N] + A[M,K] @ B[N,K]^T, with the fine-grained scales
 * applied per K-group (docsearch section 4; README "Interfaces > Notices").
 *   a    [M][K]   E4M3, row-major (K contiguous)
 *   sfa  [ceil(K/512)][align4(M)] packed UE8M0, one scale per row per K-group
 *   b    [N][K]   E4M3, row-major (K contiguous)
 *   sfb  [ceil(K/512)][align4(ceil(N/128))] packed UE8M0, one scale per 128x128 block
 *   c    [M][N]   FP32 or NULL; needs d_dtype == FG_F32; may equal d
 *   d    [M][N]   BF16 or FP32 (d_dtype)
 * M >= 0 (M == 0 returns FG_OK), K >= 128 and K % 128 == 0, N >= 16 and N % 16 == 0.
 */
int fg_fp8_gemm_nt(int M, int N, int K,
                   const uint8_t* a, const int32_t* sfa,
                   const uint8_t* b, const int32_t* sfb,
                   const float* c, void* d, int d_dtype, fg_stream_t stream);

/*
 * The other dense layouts (docsearch section 4 "Memory Layouts": SM100 supports NT, TN,
 * NN and TT; section 9 item 1, fp8_gemm_{nt, nn, tn, tt}).  The same product
 *   D[m,n] = C[m,n] + sum_k A(m,k) * B(k,n) with the same scales and C/D as the NT GEMM,
 * with the operands stored as
 *   NN:  a [M][K] (K contiguous),  b [K][N] (N contiguous)
 *   TN:  a [K][M] (M contiguous),  b [K][N] (N contiguous)
 *   TT:  a [K][M] (M contiguous),  b [N][K] (K contiguous)
 * The letter says whether the operand is stored transposed relative to the NT form's
 * A [M][K] and B^T = [N][K].  sfa and sfb keep the NT layouts (one scale per row of A
 * and 1x128 K-group; one per 128x128 block of B) whatever the operand layout.
 * Shapes as for fg_fp8_gemm_nt, plus M % 16 == 0 when A is stored [K][M] (TN, TT).
 */
int fg_fp8_gemm_nn(int M, int N, int K,
                   const uint8_t* a, const int32_t* sfa,
                   const uint8_t* b, const int32_t* sfb,
                   const float* c, void* d, int d_dtype, fg_stream_t stream);
int fg_fp8_gemm_tn(int M, int N, int K,
                   const uint8_t* a, const int32_t* sfa,
                   const uint8_t* b, const int32_t* sfb,
                   const float* c, void* d, int d_dtype, fg_stream_t stream);
int fg_fp8_gemm_tt(int M, int N, int K,
                   const uint8_t* a, const int32_t* sfa,
                   const uint8_t* b, const int32_t* sfb,
                   const float* c, void* d, int d_dtype, fg_stream_t stream);

/*
 * M-grouped contiguous NT GEMM (docsearch section 9 item 2; README "Grouped GEMMs
 * (contiguous layout)"): the token rows of all groups (experts) are concatenated
 * along M, every group segment aligned to fg_get_mk_alignment_for_contiguous_layout()
 * rows.  Row m uses the weights of group m_indices[m]:
 *   D[m,:] = A[m,:] @ B[m_indices[m]]^T
 *   a          [M_total][K] E4M3;  sfa [ceil(K/512)][align4(M_total)]
 *   b          [G][N][K]    E4M3;  sfb [G][ceil(K/512)][align4(ceil(N/128))]
 *   m_indices  [M_total] int32 on the device: group id in [0,G), or -1 for padding
 *   d          [M_total][N] BF16 or FP32
 * Rows with m_indices == -1 are neither computed into D nor written.  Within each
 * 128-row block all non-padding rows must name one group; a block whose first row is
 * -1 is skipped.  A row naming another group, or a group id >= G, is a device
 * contract violation: that row (or block) is left unwritten and the status word is set.
 * M_total % 128 == 0, G >= 1.  No C operand.
 */
int fg_m_grouped_fp8_gemm_nt_contiguous(int M_total, int N, int K, int G,
                                        const uint8_t* a, const int32_t* sfa,
                                        const uint8_t* b, const int32_t* sfb,
                                        const int32_t* m_indices,
                                        void* d, int d_dtype, fg_stream_t stream);

/*
 * Gate-up GEMM of the MoE MLP with the SwiGLU and the FP8 requantisation of its output
 * fused into the epilogue (the MoE MLP's linear 1 -> SwiGLU -> FP8 cast for linear 2:
 * "Mega MoE", docsearch / README; MegaMoE DCU README "Runtime Routing", K2 "SwiGLU +
 * channelwise FP8 quant").  Each group's weight b[g] holds I gate rows then I up rows:
 *   h = A[m,:] @ b[g]^T  (g = m_indices[m]),   y[i] = SiLU(h[i]) * h[I + i],
 *   SiLU(x) = x / (1 + exp(-x)),
 * then per row and 1x128 group of y: scale 2^e, the smallest with amax <= 448 * 2^e, and
 * q = E4M3 round-to-nearest-even of y * 2^-e (computed in FP32): exactly the A operand
 * (and its sfa) of the down projection.
 *   a    [M_total][K] E4M3, sfa [ceil(K/512)][align4(M_total)]
 *   b    [G][2I][K]   E4M3, sfb [G][ceil(K/512)][align4(2I/128)] (128x128 blocks)
 *   q    [M_total][I] E4M3 (out), sfq [ceil(I/512)][align4(M_total)] packed UE8M0 (out)
 * Padding rows (m_indices == -1) are left untouched in q and sfq; only the bytes of sfq
 * that name a computed group are written (the caller zeroes the rest if it reads them).
 * I >= 128 and I % 128 == 0; the rest as fg_m_grouped_fp8_gemm_nt_contiguous.
 */
int fg_m_grouped_fp8_gemm_nt_contiguous_swiglu(int M_total, int I, int K, int G,
                                               const uint8_t* a, const int32_t* sfa,
                                               const uint8_t* b, const int32_t* sfb,
                                               const int32_t* m_indices,
                                               uint8_t* q, int32_t* sfq, fg_stream_t stream);

/* The same fused gate-up GEMM for the masked layout: a [G][M_max][K] with
 * sfa [G][ceil(K/512)][align4(M_max)], b and sfb as above, masked_m as for
 * fg_m_grouped_fp8_gemm_nt_masked; q [G][M_max][I], sfq [G][ceil(I/512)][align4(M_max)];
 * rows >= masked_m[g] are left untouched. */
int fg_m_grouped_fp8_gemm_nt_masked_swiglu(int G, int M_max, int I, int K,
                                           const uint8_t* a, const int32_t* sfa,
                                           const uint8_t* b, const int32_t* sfb,
                                           const int32_t* masked_m,
                                           uint8_t* q, int32_t* sfq, fg_stream_t stream);

/*
 * The same M-grouped contiguous GEMM with each group's weights stored N-major
 * (docsearch section 9 item 2, m_grouped_fp8_gemm_{nt, nn}_contiguous):
 *   D[m,:] = A[m,:] @ B[m_indices[m]],  b [G][K][N] E4M3 (N contiguous)
 * Everything else (sfa, sfb, m_indices, d, padding rows, contract checks) as for
 * fg_m_grouped_fp8_gemm_nt_contiguous.
 */
int fg_m_grouped_fp8_gemm_nn_contiguous(int M_total, int N, int K, int G,
                                        const uint8_t* a, const int32_t* sfa,
                                        const uint8_t* b, const int32_t* sfb,
                                        const int32_t* m_indices,
                                        void* d, int d_dtype, fg_stream_t stream);

/*
 * M-grouped masked NT GEMM (docsearch section 9 item 4; README "Grouped GEMMs (masked
 * layout)"): group g owns rows [0, M_max) of its slice; only rows m < masked_m[g]
 * are valid.  The counts live on the device, so the call needs no host knowledge of
 * them and can sit inside a CUDA graph:
 *   D[g, m, :] = A[g, m, :] @ B[g]^T        for m < masked_m[g]
 *   a         [G][M_max][K] E4M3;  sfa [G][ceil(K/512)][align4(M_max)]
 *   b         [G][N][K]     E4M3;  sfb [G][ceil(K/512)][align4(ceil(N/128))]
 *   masked_m  [G] int32 on the device, each in [0, M_max]
 *   expected_m  host hint of the typical masked_m (tile-size choice only; <= 0: none);
 *               results never depend on it
 *   d         [G][M_max][N] BF16 or FP32
 * Rows m >= masked_m[g] are never written, and their A rows (which may hold any bytes,
 * NaN codes included) never reach a valid row.  A mask outside [0, M_max] is clamped
 * and recorded as a device contract violation.  1 <= G <= 256, M_max >= 1.  No C operand.
 */
int fg_m_grouped_fp8_gemm_nt_masked(int G, int M_max, int N, int K,
                                    const uint8_t* a, const int32_t* sfa,
                                    const uint8_t* b, const int32_t* sfb,
                                    const int32_t* masked_m, int expected_m,
                                    void* d, int d_dtype, fg_stream_t stream);

/*
 * K-grouped contiguous TN GEMM, the MoE weight gradient (docsearch section 9 item 3;
 * README "Grouped GEMMs (contiguous layout)", last paragraph): M and N are fixed,
 * and group g owns the K rows [off_g, off_g + ks[g]) of both operands:
 *   D[g] = C[g] + A[off_g : off_g+ks[g], :]^T @ B[off_g : off_g+ks[g], :]
 *   a    [K_total][M] E4M3 (M contiguous: MN-major)
 *   sfa  [ceil(K_total/512)][align4(M)] packed UE8M0, 1x128 along K per column m
 *   b    [K_total][N] E4M3 (N contiguous)
 *   sfb  [ceil(K_total/512)][align4(N)] packed UE8M0, 1x128 along K per column n
 *   ks   [G] int32 on the device; each a multiple of 128 (0 allowed); sum == K_total
 *   c    [G][M][N] FP32 or NULL (NULL: C = 0); may equal d
 *   d    [G][M][N] FP32
 * Scale groups are counted over the concatenated K axis (group of element k is k/128),
 * so no group straddles two segments.  A ks that breaks these rules is a device
 * contract violation: nothing is written and the status word is set.
 * 1 <= G <= 256, K_total % 128 == 0, M >= 16 and M % 16 == 0, N % 16 == 0.
 */
int fg_k_grouped_fp8_gemm_tn_contiguous(int G, int M, int N, int K_total,
                                        const uint8_t* a, const int32_t* sfa,
                                        const uint8_t* b, const int32_t* sfb,
                                        const int32_t* ks, const float* c, float* d,
                                        fg_stream_t stream);

/*
 * FP8 x FP4 GEMMs: E4M3 activations times FP4 weights.  The pages name an FP8xFP4 GEMM
 * (Korean README translation, news of 2026.04.16; yuguo-Jack/DeepGEMM README, "News") and
 * give the Mega MoE's linear layers as FP8 x FP4 with weights in "FP4 with UE8M0 SF"
 * (Chinese post, "Mega MoE": mma_type 'fp8xfp4'; same README, "CUDA Mega MoE").  Each call
 * computes what its FP8 counterpart above computes, with B read as:
 *   - FP4 = E2M1 (OCP Microscaling element: sign, 2 exponent bits with bias 1, 1 mantissa
 *     bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; no inf or NaN), two codes per byte along
 *     K: element 2i in bits 0-3, 2i+1 in bits 4-7.  b is [N][K/2] bytes ([G][N][K/2]).
 *   - one UE8M0 scale per 32 consecutive K elements of each row of B (the MXFP4 block),
 *     packed four per int32 (byte j of word w = block 4w+j, i.e. one word per row and
 *     128-wide K-group), MN-major: sfb [K/128][align4(N)] int32 ([G][K/128][align4(N)]).
 * a, sfa, c, d, m_indices, masked_m, expected_m, the shape rules, the device contract and
 * the status reporting are those of fg_fp8_gemm_nt, fg_m_grouped_fp8_gemm_nt_contiguous and
 * fg_m_grouped_fp8_gemm_nt_masked.  b must be 32-byte aligned (FG_ERR_INVALID_ARG
 * otherwise).  The accumulation is FP32 in the tensor core with both scales applied per
 * 32-wide K step.
 */
int fg_fp8_fp4_gemm_nt(int M, int N, int K,
                       const uint8_t* a, const int32_t* sfa,
                       const uint8_t* b, const int32_t* sfb,
                       const float* c, void* d, int d_dtype, fg_stream_t stream);
int fg_m_grouped_fp8_fp4_gemm_nt_contiguous(int M_total, int N, int K, int G,
                                            const uint8_t* a, const int32_t* sfa,
                                            const uint8_t* b, const int32_t* sfb,
                                            const int32_t* m_indices,
                                            void* d, int d_dtype, fg_stream_t stream);
int fg_m_grouped_fp8_fp4_gemm_nt_masked(int G, int M_max, int N, int K,
                                        const uint8_t* a, const int32_t* sfa,
                                        const uint8_t* b, const int32_t* sfb,
                                        const int32_t* masked_m, int expected_m,
                                        void* d, int d_dtype, fg_stream_t stream);
/* The fused gate-up GEMMs with FP4 weights (the Mega MoE's linear 1 in FP8 x FP4, then
 * SwiGLU and the requantisation for linear 2): fg_m_grouped_fp8_gemm_nt_{contiguous,
 * masked}_swiglu with b [G][2I][K/2] packed E2M1 (I gate rows, then I up rows) and
 * sfb [G][K/128][align4(2I)] (one scale per 32 K elements of a row); everything else,
 * q and sfq included, as for the E4M3-weight calls.  b must be 32-byte aligned. */
int fg_m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(int M_total, int I, int K, int G,
                                                   const uint8_t* a, const int32_t* sfa,
                                                   const uint8_t* b, const int32_t* sfb,
                                                   const int32_t* m_indices, uint8_t* q, int32_t* sfq,
                                                   fg_stream_t stream);
int fg_m_grouped_fp8_fp4_gemm_nt_masked_swiglu(int G, int M_max, int I, int K,
                                               const uint8_t* a, const int32_t* sfa,
                                               const uint8_t* b, const int32_t* sfb,
                                               const int32_t* masked_m, uint8_t* q, int32_t* sfq,
                                               fg_stream_t stream);

/*
 * FP32 -> E4M3 quantisation with UE8M0 scales, written straight into the packed,
 * MN-major, TMA-aligned scale layout the GEMMs above read.  The pages leave the FP8
 * cast to the user and list layout helpers for it ("DeepGEMM Documentation", section
 * 4 note on FP8 casting; section 10: transform_sf_into_required_layout,
 * get_mn_major_tma_aligned_packed_ue8m0_tensor,
 * get_k_grouped_mn_major_tma_aligned_packed_ue8m0_tensor).
 * Scale of a group: the smallest power of two 2^e with amax <= 448 * 2^e, stored as
 * the byte e + 127 (clamped to [0, 254]; an all-zero group gets 127); code: E4M3
 * round-to-nearest-even of x * 2^-e.  Bytes of missing tail groups in the last packed
 * word are 0; the MN padding words of `sf` are not written.
 * All arrays are device pointers, 16-byte aligned; asynchronous on `stream`.
 */
/* x [rows][K] FP32 -> q [rows][K] E4M3, sf [ceil(K/512)][align4(rows)] (1x128 groups
 * along K per row: the activation scales of every NT GEMM).  K % 128 == 0. */
int fg_quantize_1x128_rows(int rows, int K, const float* x, uint8_t* q, int32_t* sf,
                           fg_stream_t stream);

/* w [G][N][K] FP32 -> q [G][N][K] E4M3, sf [G][ceil(K/512)][align4(ceil(N/128))]
 * (one scale per 128x128 block: the weight scales of the NT GEMMs).  K % 128 == 0; a
 * ragged last row block takes its scale from its valid rows. */
int fg_quantize_128x128_blocks(int G, int N, int K, const float* w, uint8_t* q, int32_t* sf,
                               fg_stream_t stream);

/* x [K][MN] FP32 -> q [K][MN] E4M3, sf [ceil(K/512)][align4(MN)] (1x128 groups along
 * the leading K axis per column: both operands of the K-grouped GEMM; with zero-padded
 * segments the packing is the K-grouped one).  K % 128 == 0, MN % 16 == 0. */
int fg_quantize_1x128_cols(int K, int MN, const float* x, uint8_t* q, int32_t* sf,
                           fg_stream_t stream);

/* w [G][N][K] FP32 -> q [G][N][K/2] packed E2M1 (element 2i in bits 0-3 of byte i) and
 * sf [G][K/128][align4(N)] int32: the FP4 weights of the FP8 x FP4 GEMMs, one UE8M0 scale
 * per 32 K elements of a row, four per word.  Scale of a block: the smallest power of two
 * 2^e with amax <= 6 * 2^e (byte e + 127, clamped to [0, 254]; an all-zero block gets 127);
 * code: E2M1 round-to-nearest-even of x * 2^-e (ties to the even mantissa).  K % 128 == 0;
 * every word of sf's [K/128][N] part is written, its padding words are not. */
int fg_quantize_mxfp4(int G, int N, int K, const float* w, uint8_t* q, int32_t* sf, fg_stream_t stream);

/*
 * MQA logits of the lightning indexer, non-paged (docsearch section 11 "Use V3.2 MQA
 * Kernels for Indexers", fp8_mqa_logits): for query token i and every kv token j in
 * [ks[i], ke[i]) (clipped to [0, T)),
 *   out[i, j] = sum_h relu(q[i, h, :] . (kv[j, :] * kv_sf[j])) * weights[i, h]
 * computed with FP32 accumulation; with clean_logits != 0 every other entry of out is
 * -inf, otherwise those entries are left untouched.
 *   q        [S][H][D]  E4M3          kv       [T][D] E4M3      kv_sf [T] FP32
 *   weights  [S][H]     FP32          ks, ke   [S] int32 (device)
 *   out      [S][T]     FP32
 * Supported: H == 64 and D == 128 (FG_ERR_UNSUPPORTED otherwise); S >= 0, T >= 1.
 */
int fg_fp8_mqa_logits(int S, int T, int H, int D, const uint8_t* q, const uint8_t* kv,
                      const float* kv_sf, const float* weights, const int32_t* ks,
                      const int32_t* ke, int clean_logits, float* out, fg_stream_t stream);

/* Row alignment of each group segment in the contiguous layout: 128, the M block
 * (docsearch section 9 item 2 and section 10). */
int fg_get_mk_alignment_for_contiguous_layout(void);

/* x rounded up so that x * elem_bytes is a multiple of 16 bytes (section 10,
 * get_tma_aligned_size).  Returns -1 for elem_bytes not in {1,2,4,8} or x < 0. */
int fg_get_tma_aligned_size(int x, int elem_bytes);

/* Maximum number of SMs the persistent kernels use (section 10, set/get_num_sms).
 * n <= 0 restores the default (all SMs of the current device).  get returns the value
 * in force for the current device, or -1 when no device is available. */
void fg_set_num_sms(int n);
int fg_get_num_sms(void);

/* Programmatic dependent launch of the GEMM kernels (section 10, set_pdl/get_pdl).
 * Enabled (the default), every GEMM is launched so that it may begin while the previous
 * kernel of the stream is still finishing: its CTAs initialise barriers and tensor
 * memory, then wait until the previous grid has completed and its writes are visible
 * before touching global memory (so results never depend on the setting); and each GEMM
 * allows the next programmatic launch to begin as soon as all of its CTAs are running.
 * enable = 0 launches with plain stream ordering. */
void fg_set_pdl(int enable);
int fg_get_pdl(void);

/* Reads and clears the device status word of the current device after the work queued
 * on `stream` so far, then synchronises `stream`: returns FG_OK, FG_ERR_DEVICE_CONTRACT
 * or FG_ERR_DEVICE_TIMEOUT (the first event since the last read), or FG_ERR_CUDA if a
 * CUDA call failed.  *detail (may be NULL) receives the raw code:
 *   0x101  a contiguous m_indices entry names a group >= G
 *   0x102  a contiguous 128-row block mixes groups (a row names another group than the
 *          block's first row, or a block whose first row is -1 names a group later on)
 *   0x103  a masked_m entry lies outside [0, M_max]
 *   0x104  K-grouped ks entries negative, not multiples of 128, or not summing to K_total
 *   0x105  internal: a split-K launch without one tile per cluster
 *   0x2xx  a bounded wait inside a kernel ran out (xx says which role waited)
 * The word is one per device and shared by every stream: a kernel of another stream that
 * records an event concurrently is reported by this call or by the next one (the read
 * and the clear are a single atomic exchange, so no event is lost).  Calls from several
 * host threads are serialised. */
int fg_get_device_error(fg_stream_t stream, int* detail);

/* Static description of a status code. */
const char* fg_status_string(int status);

/* Test hook for the time-out path: while enabled, the next GEMM launches have their
 * operand producer skip its first stage, so the MMA issuer's bounded wait runs out
 * after timeout_us microseconds, the kernel records FG_ERR_DEVICE_TIMEOUT and every
 * role exits cleanly.  enable = 0 restores normal operation and the default time-out. */
void fg_debug_inject_stall(int enable, uint32_t timeout_us);

#ifdef __cplusplus
}
#endif

#endif /* FG_H */
