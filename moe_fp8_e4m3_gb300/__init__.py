"""Python binding of the fine-grained FP8 GEMM C-ABI library (``include/fg.h``).

Argument marshalling only: every function takes torch CUDA tensors, checks dtypes and
contiguity, and passes raw device pointers, host-side sizes and the current CUDA stream
to the same-named ``fg_*`` C entry point.  All arithmetic runs in the library's CUDA
kernels; there is no fallback.  Importing fails loudly if ``libfg.so`` has not been
built (``moe_fp8_e4m3_gb300.build.build()``)."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfg.so")

FG_OK = 0
FG_ERR_INVALID_ARG = -1
FG_ERR_UNSUPPORTED = -2
FG_ERR_CUDA = -3
FG_ERR_DEVICE_CONTRACT = -4
FG_ERR_DEVICE_TIMEOUT = -5
FG_BF16 = 0
FG_F32 = 1

_P = ctypes.c_void_p
_I = ctypes.c_int

_SIGNATURES = {
    "fg_fp8_gemm_nt": (_I, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    "fg_fp8_gemm_nn": (_I, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    "fg_fp8_gemm_tn": (_I, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    "fg_fp8_gemm_tt": (_I, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    "fg_m_grouped_fp8_gemm_nt_contiguous": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    "fg_m_grouped_fp8_gemm_nn_contiguous": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    "fg_m_grouped_fp8_gemm_nt_contiguous_swiglu": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "fg_fp8_mqa_logits": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "fg_m_grouped_fp8_gemm_nt_masked_swiglu": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "fg_m_grouped_fp8_gemm_nt_masked": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _I, _P]),
    "fg_fp8_fp4_gemm_nt": (_I, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    "fg_m_grouped_fp8_fp4_gemm_nt_contiguous": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    "fg_m_grouped_fp8_fp4_gemm_nt_masked": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _I, _P]),
    "fg_m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "fg_m_grouped_fp8_fp4_gemm_nt_masked_swiglu": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "fg_k_grouped_fp8_gemm_tn_contiguous": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "fg_quantize_1x128_rows": (_I, [_I, _I, _P, _P, _P, _P]),
    "fg_quantize_128x128_blocks": (_I, [_I, _I, _I, _P, _P, _P, _P]),
    "fg_quantize_1x128_cols": (_I, [_I, _I, _P, _P, _P, _P]),
    "fg_quantize_mxfp4": (_I, [_I, _I, _I, _P, _P, _P, _P]),
    "fg_get_mk_alignment_for_contiguous_layout": (_I, []),
    "fg_get_tma_aligned_size": (_I, [_I, _I]),
    "fg_set_num_sms": (None, [_I]),
    "fg_get_num_sms": (_I, []),
    "fg_set_pdl": (None, [_I]),
    "fg_get_pdl": (_I, []),
    "fg_get_device_error": (_I, [_P, ctypes.POINTER(_I)]),
    "fg_status_string": (ctypes.c_char_p, [_I]),
    "fg_debug_inject_stall": (None, [_I, ctypes.c_uint32]),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class FgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.fg_status_string(status).decode()} (status {status})")


def _check(status: int, where: str) -> None:
    if status != FG_OK:
        raise FgError(status, where)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _fp8(t, name):
    import torch
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or not t.is_contiguous() or not t.is_cuda:
        raise TypeError(f"{name} must be a contiguous CUDA uint8/float8_e4m3fn tensor")


def _i32(t, name):
    import torch
    if t.dtype != torch.int32 or not t.is_contiguous() or not t.is_cuda:
        raise TypeError(f"{name} must be a contiguous CUDA int32 tensor")


def _out(t, name):
    import torch
    if t.dtype not in (torch.bfloat16, torch.float32) or not t.is_contiguous() or not t.is_cuda:
        raise TypeError(f"{name} must be a contiguous CUDA bfloat16/float32 tensor")
    return FG_F32 if t.dtype == torch.float32 else FG_BF16


def _c(t):
    import torch
    if t is not None and (t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda):
        raise TypeError("c must be a contiguous CUDA float32 tensor")


def fp8_gemm_nt(a, sfa, b, sfb, d, c=None, stream=None) -> None:
    """D = C + A @ B.T.  a [M,K], b [N,K] E4M3; sfa [ceil(K/512), align4(M)] and
    sfb [ceil(K/512), align4(ceil(N/128))] packed UE8M0 int32; d [M,N] BF16/FP32;
    c optional FP32 [M,N] (FP32 d only; may be d)."""
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _c(c)
    code = _out(d, "d")
    m, k = a.shape
    n = b.shape[0]
    _check(lib.fg_fp8_gemm_nt(m, n, k, _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d),
                              code, _stream(stream)), "fp8_gemm_nt")


def _dense_layout(fn, name, a, sfa, b, sfb, d, c, stream, a_t, b_n):
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _c(c)
    code = _out(d, "d")
    k, m = a.shape if a_t else a.shape[::-1]
    n = b.shape[1] if b_n else b.shape[0]
    _check(fn(m, n, k, _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d), code, _stream(stream)), name)


def fp8_gemm_nn(a, sfa, b, sfb, d, c=None, stream=None) -> None:
    """D = C + A @ B.  a [M,K], b [K,N] E4M3 (N contiguous); scales, c and d as fp8_gemm_nt."""
    _dense_layout(lib.fg_fp8_gemm_nn, "fp8_gemm_nn", a, sfa, b, sfb, d, c, stream, False, True)


def fp8_gemm_tn(a, sfa, b, sfb, d, c=None, stream=None) -> None:
    """D = C + A.T @ B.  a [K,M] (M contiguous, M % 16 == 0), b [K,N]; scales, c and d as fp8_gemm_nt."""
    _dense_layout(lib.fg_fp8_gemm_tn, "fp8_gemm_tn", a, sfa, b, sfb, d, c, stream, True, True)


def fp8_gemm_tt(a, sfa, b, sfb, d, c=None, stream=None) -> None:
    """D = C + A.T @ B.T.  a [K,M] (M contiguous, M % 16 == 0), b [N,K]; scales, c and d as fp8_gemm_nt."""
    _dense_layout(lib.fg_fp8_gemm_tt, "fp8_gemm_tt", a, sfa, b, sfb, d, c, stream, True, False)


def m_grouped_fp8_gemm_nn_contiguous(a, sfa, b, sfb, m_indices, d, stream=None) -> None:
    """D[m] = A[m] @ B[m_indices[m]] for rows with m_indices[m] >= 0.  a [M_total,K];
    b [G,K,N] (N contiguous); sfb [G, ceil(K/512), align4(ceil(N/128))]; m_indices int32 [M_total]."""
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _i32(m_indices, "m_indices")
    code = _out(d, "d")
    m_total, k = a.shape
    g, _, n = b.shape
    _check(lib.fg_m_grouped_fp8_gemm_nn_contiguous(m_total, n, k, g, _ptr(a), _ptr(sfa), _ptr(b),
                                                   _ptr(sfb), _ptr(m_indices), _ptr(d), code,
                                                   _stream(stream)), "m_grouped_fp8_gemm_nn_contiguous")


def m_grouped_fp8_gemm_nt_contiguous_swiglu(a, sfa, b, sfb, m_indices, q, sfq, stream=None) -> None:
    """Gate-up GEMM + SwiGLU + per-1x128 FP8 requantisation.  a [M_total,K]; b [G,2I,K]
    (I gate rows, then I up rows); q [M_total,I] uint8 (E4M3 codes, out);
    sfq [ceil(I/512), align4(M_total)] int32 packed UE8M0 (out)."""
    _fp8(a, "a"); _fp8(b, "b"); _fp8(q, "q"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _i32(sfq, "sfq")
    _i32(m_indices, "m_indices")
    m_total, k = a.shape
    g, n2, _ = b.shape
    _check(lib.fg_m_grouped_fp8_gemm_nt_contiguous_swiglu(m_total, n2 // 2, k, g, _ptr(a), _ptr(sfa), _ptr(b),
                                                          _ptr(sfb), _ptr(m_indices), _ptr(q), _ptr(sfq),
                                                          _stream(stream)), "m_grouped_fp8_gemm_nt_contiguous_swiglu")


def m_grouped_fp8_gemm_nt_masked_swiglu(a, sfa, b, sfb, masked_m, q, sfq, stream=None) -> None:
    """The masked-layout gate-up GEMM + SwiGLU + requantisation.  a [G,M_max,K]; b [G,2I,K];
    q [G,M_max,I] uint8 (out); sfq [G, ceil(I/512), align4(M_max)] int32 (out)."""
    _fp8(a, "a"); _fp8(b, "b"); _fp8(q, "q"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _i32(sfq, "sfq")
    _i32(masked_m, "masked_m")
    g, m_max, k = a.shape
    n2 = b.shape[1]
    _check(lib.fg_m_grouped_fp8_gemm_nt_masked_swiglu(g, m_max, n2 // 2, k, _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb),
                                                      _ptr(masked_m), _ptr(q), _ptr(sfq), _stream(stream)),
           "m_grouped_fp8_gemm_nt_masked_swiglu")


def fp8_mqa_logits(q, kv, kv_sf, weights, ks, ke, out, clean_logits=True, stream=None) -> None:
    """Lightning-indexer MQA logits.  q [S,H,D] E4M3 (H=64, D=128); kv [T,D] E4M3;
    kv_sf float32 [T]; weights float32 [S,H]; ks, ke int32 [S]; out float32 [S,T]."""
    import torch
    _fp8(q, "q"); _fp8(kv, "kv"); _i32(ks, "ks"); _i32(ke, "ke")
    for t, name in ((kv_sf, "kv_sf"), (weights, "weights"), (out, "out")):
        if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
            raise TypeError(f"{name} must be a contiguous CUDA float32 tensor")
    s_len, heads, dim = q.shape
    t_len = kv.shape[0]
    _check(lib.fg_fp8_mqa_logits(s_len, t_len, heads, dim, _ptr(q), _ptr(kv), _ptr(kv_sf), _ptr(weights), _ptr(ks),
                                 _ptr(ke), 1 if clean_logits else 0, _ptr(out), _stream(stream)), "fp8_mqa_logits")


def m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, m_indices, d, stream=None) -> None:
    """D[m] = A[m] @ B[m_indices[m]].T for rows with m_indices[m] >= 0.  a [M_total,K];
    b [G,N,K]; sfb [G, ceil(K/512), align4(ceil(N/128))]; m_indices int32 [M_total]."""
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _i32(m_indices, "m_indices")
    code = _out(d, "d")
    m_total, k = a.shape
    g, n, _ = b.shape
    _check(lib.fg_m_grouped_fp8_gemm_nt_contiguous(m_total, n, k, g, _ptr(a), _ptr(sfa), _ptr(b),
                                                   _ptr(sfb), _ptr(m_indices), _ptr(d), code,
                                                   _stream(stream)), "m_grouped_fp8_gemm_nt_contiguous")


def m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, masked_m, d, expected_m=0, stream=None) -> None:
    """D[g, m] = A[g, m] @ B[g].T for m < masked_m[g].  a [G,M_max,K];
    sfa [G, ceil(K/512), align4(M_max)]; b [G,N,K]; masked_m int32 [G] on the device."""
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _i32(masked_m, "masked_m")
    code = _out(d, "d")
    g, m_max, k = a.shape
    n = b.shape[1]
    _check(lib.fg_m_grouped_fp8_gemm_nt_masked(g, m_max, n, k, _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb),
                                               _ptr(masked_m), int(expected_m), _ptr(d), code,
                                               _stream(stream)), "m_grouped_fp8_gemm_nt_masked")


def _fp4(t, name):
    import torch
    ok = t.dtype == torch.uint8 or t.dtype == getattr(torch, "float4_e2m1fn_x2", torch.uint8)
    if not ok or not t.is_contiguous() or not t.is_cuda:
        raise TypeError(f"{name} must be a contiguous CUDA uint8/float4_e2m1fn_x2 tensor of packed E2M1 pairs")


def fp8_fp4_gemm_nt(a, sfa, b, sfb, d, c=None, stream=None) -> None:
    """D = C + A @ B.T with FP4 B.  a [M,K] E4M3, sfa as fp8_gemm_nt; b [N,K/2] packed E2M1
    (element 2i in the low nibble); sfb [K/128, align4(N)] int32, one UE8M0 scale per 32 K
    elements of each row of B; d [M,N] BF16/FP32; c optional FP32 [M,N] (FP32 d only)."""
    _fp8(a, "a"); _fp4(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _c(c)
    code = _out(d, "d")
    m, k = a.shape
    n = b.shape[0]
    _check(lib.fg_fp8_fp4_gemm_nt(m, n, k, _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d),
                                  code, _stream(stream)), "fp8_fp4_gemm_nt")


def m_grouped_fp8_fp4_gemm_nt_contiguous(a, sfa, b, sfb, m_indices, d, stream=None) -> None:
    """The M-grouped contiguous GEMM with FP4 B.  a [M_total,K]; b [G,N,K/2] packed E2M1;
    sfb [G, K/128, align4(N)] int32 (1x32 blocks); m_indices int32 [M_total]."""
    _fp8(a, "a"); _fp4(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _i32(m_indices, "m_indices")
    code = _out(d, "d")
    m_total, k = a.shape
    g, n, _ = b.shape
    _check(lib.fg_m_grouped_fp8_fp4_gemm_nt_contiguous(m_total, n, k, g, _ptr(a), _ptr(sfa), _ptr(b),
                                                       _ptr(sfb), _ptr(m_indices), _ptr(d), code,
                                                       _stream(stream)), "m_grouped_fp8_fp4_gemm_nt_contiguous")


def m_grouped_fp8_fp4_gemm_nt_masked(a, sfa, b, sfb, masked_m, d, expected_m=0, stream=None) -> None:
    """The M-grouped masked GEMM with FP4 B.  a [G,M_max,K]; b [G,N,K/2] packed E2M1;
    sfb [G, K/128, align4(N)] int32 (1x32 blocks); masked_m int32 [G] on the device."""
    _fp8(a, "a"); _fp4(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _i32(masked_m, "masked_m")
    code = _out(d, "d")
    g, m_max, k = a.shape
    n = b.shape[1]
    _check(lib.fg_m_grouped_fp8_fp4_gemm_nt_masked(g, m_max, n, k, _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb),
                                                   _ptr(masked_m), int(expected_m), _ptr(d), code,
                                                   _stream(stream)), "m_grouped_fp8_fp4_gemm_nt_masked")


def m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(a, sfa, b, sfb, m_indices, q, sfq, stream=None) -> None:
    """The fused gate-up GEMM with FP4 weights.  a [M_total,K]; b [G,2I,K/2] packed E2M1 (I gate
    rows, then I up rows); sfb [G, K/128, align4(2I)] int32 (1x32 blocks); q [M_total,I] uint8
    (out); sfq [ceil(I/512), align4(M_total)] int32 (out)."""
    _fp8(a, "a"); _fp4(b, "b"); _fp8(q, "q"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _i32(sfq, "sfq")
    _i32(m_indices, "m_indices")
    m_total, k = a.shape
    g, n2, _ = b.shape
    _check(lib.fg_m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(m_total, n2 // 2, k, g, _ptr(a), _ptr(sfa), _ptr(b),
                                                              _ptr(sfb), _ptr(m_indices), _ptr(q), _ptr(sfq),
                                                              _stream(stream)),
           "m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu")


def m_grouped_fp8_fp4_gemm_nt_masked_swiglu(a, sfa, b, sfb, masked_m, q, sfq, stream=None) -> None:
    """The masked fused gate-up GEMM with FP4 weights.  a [G,M_max,K]; b [G,2I,K/2] packed E2M1;
    sfb [G, K/128, align4(2I)]; q [G,M_max,I] uint8 (out); sfq [G, ceil(I/512), align4(M_max)]."""
    _fp8(a, "a"); _fp4(b, "b"); _fp8(q, "q"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _i32(sfq, "sfq")
    _i32(masked_m, "masked_m")
    g, m_max, k = a.shape
    n2 = b.shape[1]
    _check(lib.fg_m_grouped_fp8_fp4_gemm_nt_masked_swiglu(g, m_max, n2 // 2, k, _ptr(a), _ptr(sfa), _ptr(b),
                                                          _ptr(sfb), _ptr(masked_m), _ptr(q), _ptr(sfq),
                                                          _stream(stream)),
           "m_grouped_fp8_fp4_gemm_nt_masked_swiglu")


def k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, ks, d, c=None, stream=None) -> None:
    """D[g] = C[g] + A_g.T @ B_g.  a [K_total,M], b [K_total,N] E4M3 (MN-major);
    sfa [ceil(K_total/512), align4(M)], sfb [ceil(K_total/512), align4(N)];
    ks int32 [G] on the device; d (and c) FP32 [G,M,N]."""
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _i32(ks, "ks"); _c(c)
    if _out(d, "d") != FG_F32:
        raise TypeError("d must be float32")
    k_total, m = a.shape
    n = b.shape[1]
    g = ks.shape[0]
    _check(lib.fg_k_grouped_fp8_gemm_tn_contiguous(g, m, n, k_total, _ptr(a), _ptr(sfa), _ptr(b),
                                                   _ptr(sfb), _ptr(ks), _ptr(c), _ptr(d),
                                                   _stream(stream)), "k_grouped_fp8_gemm_tn_contiguous")


def _f32(t, name):
    import torch
    if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
        raise TypeError(f"{name} must be a contiguous CUDA float32 tensor")


def quantize_1x128_rows(x, q, sf, stream=None) -> None:
    """x [rows,K] FP32 -> q [rows,K] E4M3 bytes, sf [ceil(K/512), align4(rows)] packed UE8M0."""
    _f32(x, "x"); _fp8(q, "q"); _i32(sf, "sf")
    rows, k = x.shape
    _check(lib.fg_quantize_1x128_rows(rows, k, _ptr(x), _ptr(q), _ptr(sf), _stream(stream)),
           "quantize_1x128_rows")


def quantize_128x128_blocks(w, q, sf, stream=None) -> None:
    """w [G,N,K] (or [N,K]) FP32 -> q E4M3, sf [G, ceil(K/512), align4(ceil(N/128))]."""
    _f32(w, "w"); _fp8(q, "q"); _i32(sf, "sf")
    g, n, k = (1, *w.shape) if w.dim() == 2 else w.shape
    _check(lib.fg_quantize_128x128_blocks(g, n, k, _ptr(w), _ptr(q), _ptr(sf), _stream(stream)),
           "quantize_128x128_blocks")


def quantize_mxfp4(w, q, sf, stream=None) -> None:
    """w [G,N,K] (or [N,K]) FP32 -> q [.., N, K/2] packed E2M1, sf [G, K/128, align4(N)]
    (one UE8M0 scale per 32 K elements of a row): the FP4 weights of the FP8 x FP4 GEMMs."""
    _f32(w, "w"); _fp4(q, "q"); _i32(sf, "sf")
    g, n, k = (1, *w.shape) if w.dim() == 2 else w.shape
    _check(lib.fg_quantize_mxfp4(g, n, k, _ptr(w), _ptr(q), _ptr(sf), _stream(stream)), "quantize_mxfp4")


def quantize_1x128_cols(x, q, sf, stream=None) -> None:
    """x [K,MN] FP32 -> q [K,MN] E4M3, sf [ceil(K/512), align4(MN)] (groups along K)."""
    _f32(x, "x"); _fp8(q, "q"); _i32(sf, "sf")
    k, mn = x.shape
    _check(lib.fg_quantize_1x128_cols(k, mn, _ptr(x), _ptr(q), _ptr(sf), _stream(stream)),
           "quantize_1x128_cols")


def get_mk_alignment_for_contiguous_layout() -> int:
    return lib.fg_get_mk_alignment_for_contiguous_layout()


def get_tma_aligned_size(x: int, elem_bytes: int) -> int:
    return lib.fg_get_tma_aligned_size(x, elem_bytes)


def set_num_sms(n: int) -> None:
    lib.fg_set_num_sms(n)


def get_num_sms() -> int:
    return lib.fg_get_num_sms()


def set_pdl(enable: bool) -> None:
    """Programmatic dependent launch of the GEMM kernels on (default) or off."""
    lib.fg_set_pdl(1 if enable else 0)


def get_pdl() -> bool:
    return bool(lib.fg_get_pdl())


def get_device_error(stream=None) -> tuple[int, int]:
    """Synchronises the stream; returns (status, raw code) and clears the status word."""
    detail = ctypes.c_int(0)
    st = lib.fg_get_device_error(_stream(stream), ctypes.byref(detail))
    return st, detail.value


def debug_inject_stall(enable: bool, timeout_us: int = 0) -> None:
    lib.fg_debug_inject_stall(1 if enable else 0, timeout_us)
