"""The FP8 x FP4 GEMM: E4M3 activations with 1x128 UE8M0 scales times FP4 (E2M1)
weights with UE8M0 scales, as plain FP64 definitions.

TEST INFRASTRUCTURE (oracle): see the header of ``oracle/formats.py`` for who may
import it.  Shares no code with the CUDA library.

Sources, by page and section: the Korean README translation (molayo1419.me), news of
2026.04.16, and the yuguo-Jack/DeepGEMM README, "News": an FP8xFP4 GEMM joins the
library; the Chinese post (bittide), "Mega MoE", and the same README, "CUDA Mega MoE":
linear 1 and linear 2 of the MoE run FP8 x FP4 (``mma_type='fp8xfp4'``, the FP8 x FP8
form being the alternative), with the weights given as "FP4 with UE8M0 SF".  The product
is the FP8 GEMM's, ``D = C + A @ B.T``, with B's codes and scales read as below.

Readings where the pages are silent:

* FP4 is E2M1, the FP4 element of the OCP Microscaling (MX) formats: a sign bit, two
  exponent bits with bias 1 and one mantissa bit; exponent 0 is subnormal (m * 0.5);
  no infinity or NaN.  The magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4 and 6.
* "UE8M0 SF" of the FP4 weights is the MX block scale: one UE8M0 value per 32
  consecutive K elements of each weight row (MXFP4's block size).
* Storage of B: two codes per byte along K, element 2i in bits 0-3 and element 2i + 1
  in bits 4-7; B is [N, K/2] bytes ([G, N, K/2] for the grouped forms).
* B's scale bytes are packed four per int32 like the FP8 scales, byte j of word w being
  32-element block 4w + j (K elements 128w + 32j .. 128w + 32j + 31), MN-major and
  TMA-aligned: [K/128][align4(N)] int32 ([G][K/128][align4(N)] grouped).  So one word
  covers one 128-wide K-group of one row.
* A, its scales, the row routing of the grouped forms, C and the output rounding are
  those of the FP8 GEMM (``oracle/gemm.py``).
* MXFP4 quantiser (input preparation only): per 32-element block the scale is the
  smallest power of two s with amax / s <= 6; the code is the E2M1 round-to-nearest-even
  of x / s (ties to the even mantissa).
"""
from __future__ import annotations

import numpy as np

from .formats import K_GROUP, pack_ue8m0, ue8m0_to_f64, unpack_ue8m0
from .gemm import dequant_k_major, row_scales

E2M1_MAX = 6.0
MX_BLOCK = 32          # K elements per FP4 weight scale


# ---------------------------------------------------------------------------
# E2M1
# ---------------------------------------------------------------------------
def e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code from its fields: sign s (bit 3), exponent e (bits
    1-2, bias 1), mantissa m (bit 0).  e == 0: m * 0.5; otherwise (1 + m/2) * 2^(e-1)."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E2M1_TABLE.setflags(write=False)


def e2m1_to_f64(codes) -> np.ndarray:
    """Exact decode of 4-bit codes (one per uint8) to float64."""
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def unpack_fp4(packed) -> np.ndarray:
    """Bytes [..., K/2] -> codes [..., K]: element 2i from bits 0-3, 2i + 1 from bits 4-7."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def pack_fp4(codes) -> np.ndarray:
    """Codes [..., K] (K even) -> bytes [..., K/2], the inverse of :func:`unpack_fp4`."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def f64_to_e2m1(x) -> np.ndarray:
    """E2M1 round-to-nearest-even of float64 values (returns codes).

    At or above 1 the spacing of E2M1 values at exponent e = floor(log2|x|) is
    2^(e-1); below 1 (the subnormal 0.5 and zero) it is 0.5.  The magnitude is rounded
    to a multiple of the spacing with ties to even (np.rint: an even multiple has mantissa
    bit 0), clamped to 6, and encoded by its position among the eight non-negative
    values, which increase with the code.  Negative inputs set the sign bit."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                   # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, 0)             # values below 1 share the spacing of [1, 2)
    spacing = np.ldexp(1.0, e - 1)
    r = np.minimum(np.rint(a / spacing) * spacing, E2M1_MAX)
    code = np.searchsorted(E2M1_TABLE[:8], r).astype(np.int64)
    code = np.where(np.signbit(x), code | 0x8, code)
    return code.astype(np.uint8)


def ue8m0_for_amax_fp4(amax) -> np.ndarray:
    """Scale byte of an MX block whose largest magnitude is ``amax``: the smallest
    power of two 2^e with amax <= 6 * 2^e, as the byte e + 127 (clamped to [0, 254]);
    amax == 0 gives 127.  The log2 estimate is fixed up by exact comparisons."""
    amax = np.asarray(amax, dtype=np.float64)
    safe = np.where(amax > 0, amax, 1.0)
    e = np.ceil(np.log2(safe / E2M1_MAX)).astype(np.int64)
    e = np.where(safe > E2M1_MAX * np.ldexp(1.0, e), e + 1, e)
    e = np.where(safe <= E2M1_MAX * np.ldexp(1.0, e - 1), e - 1, e)
    byte = np.clip(e + 127, 0, 254)
    return np.where(amax > 0, byte, 127).astype(np.uint8)


def quantize_mxfp4(w: np.ndarray):
    """Per 32-element block along the last axis: w[N, K] -> (packed codes uint8[N, K/2],
    scale bytes uint8[N, K/32]).  K must be a multiple of 128."""
    w = np.asarray(w, dtype=np.float64)
    n, k = w.shape
    assert k % K_GROUP == 0
    blk = w.reshape(n, k // MX_BLOCK, MX_BLOCK)
    sf = ue8m0_for_amax_fp4(np.abs(blk).max(axis=2))
    q = f64_to_e2m1(blk / ue8m0_to_f64(sf)[:, :, None]).reshape(n, k)
    return pack_fp4(q), sf


def mx_scales(sfb_words: np.ndarray, n: int, k: int) -> np.ndarray:
    """Per-row, per-32-block scale bytes [n, k/32] from the packed words."""
    return unpack_ue8m0(sfb_words, n, k // MX_BLOCK)


def dequant_mxfp4(packed: np.ndarray, sf_bytes: np.ndarray) -> np.ndarray:
    """packed[R, K/2] E2M1 with sf_bytes[R, K/32] -> float64 [R, K]."""
    codes = unpack_fp4(packed)
    r, k = codes.shape
    assert sf_bytes.shape == (r, k // MX_BLOCK), (sf_bytes.shape, codes.shape)
    return e2m1_to_f64(codes) * np.repeat(ue8m0_to_f64(sf_bytes), MX_BLOCK, axis=1)


def pack_mx_scales(sf_bytes: np.ndarray) -> np.ndarray:
    """Scale bytes [N, K/32] -> packed words [K/128][align4(N)] (four blocks a word)."""
    return pack_ue8m0(sf_bytes)


# ---------------------------------------------------------------------------
# The GEMMs
# ---------------------------------------------------------------------------
def fp8_fp4_gemm_nt(a, sfa_words, b, sfb_words, c=None, rows=None) -> np.ndarray:
    """Exact-in-FP64 D = C + A @ B.T with FP4 B.

    a: uint8 [M, K] E4M3; sfa_words: int32 [ceil(K/512)][align4(M)];
    b: uint8 [N, K/2] packed E2M1; sfb_words: int32 [K/128][align4(N)];
    c: optional float32 [M, N].  Returns float64 [len(rows), N]."""
    m, k = a.shape
    n = b.shape[0]
    rows = np.arange(m) if rows is None else np.asarray(rows)
    sa = row_scales(sfa_words, m, k)[rows]
    d = dequant_k_major(a[rows], sa) @ dequant_mxfp4(b, mx_scales(sfb_words, n, k)).T
    if c is not None:
        d = d + np.asarray(c, dtype=np.float64)[rows]
    return d


def m_grouped_fp8_fp4_gemm_nt_contiguous(a, sfa_words, b, sfb_words, m_indices, rows=None):
    """a: uint8 [M_total, K]; b: uint8 [G, N, K/2]; sfb_words: int32 [G][K/128][align4(N)];
    m_indices: int32 [M_total] (expert id, or -1 for padding).

    Returns (d float64 [len(rows), N], written bool [len(rows)]) as the FP8 form does."""
    m_total, k = a.shape
    g_count, n, _ = b.shape
    rows = np.arange(m_total) if rows is None else np.asarray(rows)
    m_indices = np.asarray(m_indices)
    sa = row_scales(sfa_words, m_total, k)
    d = np.full((len(rows), n), np.nan)
    written = m_indices[rows] >= 0
    for e in range(g_count):
        sel = np.nonzero(m_indices[rows] == e)[0]
        if len(sel) == 0:
            continue
        src = rows[sel]
        be = dequant_mxfp4(b[e], mx_scales(sfb_words[e], n, k))
        d[sel] = dequant_k_major(a[src], sa[src]) @ be.T
    return d, written


def m_grouped_fp8_fp4_gemm_nt_masked(a, sfa_words, b, sfb_words, masked_m, experts=None, rows=None):
    """a: uint8 [G, M_max, K]; b: uint8 [G, N, K/2]; sfb_words: int32 [G][K/128][align4(N)].

    Returns {g: float64 [masked_m[g], N]} (or the rows asked for) as the FP8 form does."""
    g_count, m_max, k = a.shape
    n = b.shape[1]
    out = {}
    for e in (range(g_count) if experts is None else experts):
        valid = int(masked_m[e])
        sel = np.arange(max(valid, 0)) if rows is None else np.asarray(rows[e], dtype=np.int64)
        assert np.all(sel < valid), "rows beyond the mask are not computed"
        if len(sel) == 0:
            out[e] = np.zeros((0, n))
            continue
        sa = row_scales(sfa_words[e], m_max, k)[sel]
        be = dequant_mxfp4(b[e], mx_scales(sfb_words[e], n, k))
        out[e] = dequant_k_major(a[e, sel], sa) @ be.T
    return out


# ---------------------------------------------------------------------------
# Gate-up GEMM with FP4 weights + SwiGLU + per-1x128 requantisation
# ---------------------------------------------------------------------------
def m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(a, sfa_words, b, sfb_words, m_indices, rows=None):
    """The Mega MoE linear 1 in FP8 x FP4 (zh post "Mega MoE": linear 1 FP8xFP4, then SwiGLU)
    on one GPU: the contiguous gate-up GEMM with b [G, 2I, K/2] packed E2M1 (I gate rows,
    then I up rows; sfb_words [G][K/128][align4(2I)]), then SwiGLU and the per-1x128 E4M3
    requantisation of ``oracle.swiglu``.  Returns (codes, scale bytes, written) as the FP8
    form does."""
    from .swiglu import swiglu_quantize
    h, written = m_grouped_fp8_fp4_gemm_nt_contiguous(a, sfa_words, b, sfb_words, m_indices, rows)
    i = b.shape[1] // 2
    q = np.zeros((h.shape[0], i), np.uint8)
    sf = np.zeros((h.shape[0], i // K_GROUP), np.uint8)
    if written.any():
        q[written], sf[written] = swiglu_quantize(h[written])
    return q, sf, written


def m_grouped_fp8_fp4_gemm_nt_masked_swiglu(a, sfa_words, b, sfb_words, masked_m, experts=None):
    """The masked gate-up GEMM with FP4 weights + SwiGLU + requantisation:
    {g: (codes [masked_m[g], I], scale bytes [masked_m[g], I/128])}."""
    from .swiglu import swiglu_quantize
    d = m_grouped_fp8_fp4_gemm_nt_masked(a, sfa_words, b, sfb_words, masked_m, experts)
    out = {}
    i = b.shape[1] // 2
    for g, h in d.items():
        if h.shape[0] == 0:
            out[g] = (np.zeros((0, i), np.uint8), np.zeros((0, i // K_GROUP), np.uint8))
        else:
            out[g] = swiglu_quantize(h)
    return out
