"""The four GEMMs of the fine-grained FP8 hot path, as plain FP64 definitions.

TEST INFRASTRUCTURE (oracle): see the header of ``oracle/formats.py`` for who may
import it.  Shares no code with the CUDA library.

What is computed (docsearch section 4 "Understand DeepGEMM GEMM Naming and Layouts";
yuguo-Jack/DeepGEMM README, "Interfaces > Notices"): ``D = C + A @ B.T`` for the NT
layout, with A and B given as E4M3 bytes plus UE8M0 scales.  The scaled product is

    D[m, n] = C[m, n] + sum_g sa[m, g] * sb[n, g] * sum_{k in group g} a[m, k] * b[n, k]

where g runs over the 128-wide K groups.  Because every scale is a power of two,
multiplying each operand by its scale before the product is exact in FP64, so the
definition is evaluated as (dequantised A) @ (dequantised B).T in FP64 with a
library matmul: the same value up to FP64 rounding order.  Products of two E4M3
values are exact in FP64; the FP64 sums carry a relative error near K * 2^-53,
far below the comparison tolerance.

The grouped variants (docsearch section 9 "Use Normal and Grouped GEMM Kernels";
README "Grouped GEMMs (contiguous layout)" and "Grouped GEMMs (masked layout)"):

* M-grouped contiguous: token rows of all experts concatenated along M; row m uses
  the weights of expert ``m_indices[m]``; rows marked -1 are padding and are left as
  they were.
* M-grouped masked: expert g owns rows [0, M_max) of its buffer, of which only the
  first ``masked_m[g]`` are valid and computed; the rest are left as they were.
* K-grouped contiguous (TN, the MoE weight gradient): expert g owns K rows
  [off_g, off_g + ks[g]) of A[K_total, M] and B[K_total, N];
  D[g] = C[g] + A_g.T @ B_g.

The other dense layouts (docsearch section 4 "Memory Layouts"; section 9 item 1,
``fp8_gemm_{nt, nn, tn, tt}``, and item 2, ``m_grouped_fp8_gemm_{nt, nn}_contiguous``)
compute the same product with the operands stored differently: the first letter says
whether A is stored as [M, K] (N) or [K, M] (T), the second whether B is stored
transposed, [N, K] (T), or as [K, N] (N).  The scales keep their layouts.  Their oracle
is the NT definition applied to the operands read in that storage order.

Readings where the pages are silent: A scales are 1x128 per row; B scales are one
per 128x128 block (NT) or 1x128 per column (K-grouped); in the K-grouped layout the
scale group index is k/128 counted over the concatenated K axis; C is FP32 and only
present with an FP32 D; BF16 output is round-to-nearest-even of the exact result.
"""
from __future__ import annotations

import numpy as np

from .formats import (K_GROUP, ceil_div, e4m3_to_f64, f64_to_bf16, f64_to_f32,
                      ue8m0_to_f64, unpack_ue8m0)


# ---------------------------------------------------------------------------
# Dequantisation
# ---------------------------------------------------------------------------
def dequant_k_major(q: np.ndarray, sf_bytes: np.ndarray) -> np.ndarray:
    """q[R, K] E4M3 bytes with sf_bytes[R, K/128] -> float64 [R, K]."""
    r, k = q.shape
    assert sf_bytes.shape == (r, k // K_GROUP), (sf_bytes.shape, q.shape)
    s = np.repeat(ue8m0_to_f64(sf_bytes), K_GROUP, axis=1)
    return e4m3_to_f64(q) * s


def row_scales(sfa_words: np.ndarray, mn: int, k: int) -> np.ndarray:
    """Per-row scale bytes [mn, k/128] from the packed MN-major words."""
    return unpack_ue8m0(sfa_words, mn, k // K_GROUP)


def block_scales(sfb_words: np.ndarray, n: int, k: int) -> np.ndarray:
    """Per-row scale bytes [n, k/128] for B from the 128x128 block form
    (packed words over ceil(n/128) row blocks): row n uses block n // 128."""
    blk = unpack_ue8m0(sfb_words, ceil_div(n, K_GROUP), k // K_GROUP)
    return blk[np.arange(n) // K_GROUP]


def round_output(d: np.ndarray, out_dtype: str) -> np.ndarray:
    """'bf16' -> uint16 bit patterns; 'f32' -> float32."""
    if out_dtype == "bf16":
        return f64_to_bf16(d)
    if out_dtype == "f32":
        return f64_to_f32(d)
    raise ValueError(out_dtype)


# ---------------------------------------------------------------------------
# Dense NT: D = C + A @ B.T
# ---------------------------------------------------------------------------
def fp8_gemm_nt(a, sfa_words, b, sfb_words, c=None, rows=None) -> np.ndarray:
    """Exact-in-FP64 D for the dense NT GEMM.

    a: uint8 [M, K]; sfa_words: int32 [ceil(K/512)][align4(M)];
    b: uint8 [N, K]; sfb_words: int32 [ceil(K/512)][align4(ceil(N/128))];
    c: optional float32 [M, N].  ``rows`` selects output rows (default: all).
    Returns float64 [len(rows), N]."""
    m, k = a.shape
    n = b.shape[0]
    rows = np.arange(m) if rows is None else np.asarray(rows)
    sa = row_scales(sfa_words, m, k)[rows]
    sb = block_scales(sfb_words, n, k)
    d = dequant_k_major(a[rows], sa) @ dequant_k_major(b, sb).T
    if c is not None:
        d = d + np.asarray(c, dtype=np.float64)[rows]
    return d


def fp8_gemm_nn(a, sfa_words, b, sfb_words, c=None, rows=None) -> np.ndarray:
    """D = C + A @ B with a [M, K] and b stored [K, N]."""
    return fp8_gemm_nt(a, sfa_words, np.ascontiguousarray(b.T), sfb_words, c, rows)


def fp8_gemm_tn(a, sfa_words, b, sfb_words, c=None, rows=None) -> np.ndarray:
    """D = C + A @ B with a stored [K, M] and b stored [K, N]."""
    return fp8_gemm_nt(np.ascontiguousarray(a.T), sfa_words, np.ascontiguousarray(b.T), sfb_words, c, rows)


def fp8_gemm_tt(a, sfa_words, b, sfb_words, c=None, rows=None) -> np.ndarray:
    """D = C + A @ B with a stored [K, M] and b stored [N, K]."""
    return fp8_gemm_nt(np.ascontiguousarray(a.T), sfa_words, b, sfb_words, c, rows)


# ---------------------------------------------------------------------------
# M-grouped contiguous
# ---------------------------------------------------------------------------
def m_grouped_fp8_gemm_nt_contiguous(a, sfa_words, b, sfb_words, m_indices, rows=None):
    """a: uint8 [M_total, K]; sfa_words: [ceil(K/512)][align4(M_total)];
    b: uint8 [G, N, K]; sfb_words: int32 [G][ceil(K/512)][align4(ceil(N/128))];
    m_indices: int32 [M_total] (expert id, or -1 for padding).

    Returns (d float64 [len(rows), N], written bool [len(rows)]): rows with -1 are
    not written (their entries in ``d`` are NaN)."""
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
        be = dequant_k_major(b[e], block_scales(sfb_words[e], n, k))
        d[sel] = dequant_k_major(a[src], sa[src]) @ be.T
    return d, written


def m_grouped_fp8_gemm_nn_contiguous(a, sfa_words, b, sfb_words, m_indices, rows=None):
    """As m_grouped_fp8_gemm_nt_contiguous with b stored [G, K, N]."""
    return m_grouped_fp8_gemm_nt_contiguous(a, sfa_words, np.ascontiguousarray(np.transpose(b, (0, 2, 1))),
                                            sfb_words, m_indices, rows)


# ---------------------------------------------------------------------------
# M-grouped masked
# ---------------------------------------------------------------------------
def m_grouped_fp8_gemm_nt_masked(a, sfa_words, b, sfb_words, masked_m, experts=None, rows=None):
    """a: uint8 [G, M_max, K]; sfa_words: int32 [G][ceil(K/512)][align4(M_max)];
    b: uint8 [G, N, K]; sfb_words: int32 [G][ceil(K/512)][align4(ceil(N/128))];
    masked_m: int [G].

    Returns {g: float64 [masked_m[g], N]} for the selected experts: only rows
    m < masked_m[g] are computed; every other row of D is left as it was.
    ``rows`` (optional, {g: row indices}) restricts expert g's output to those rows, each
    below masked_m[g], in the order given."""
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
        be = dequant_k_major(b[e], block_scales(sfb_words[e], n, k))
        out[e] = dequant_k_major(a[e, sel], sa) @ be.T
    return out


# ---------------------------------------------------------------------------
# K-grouped contiguous, TN
# ---------------------------------------------------------------------------
def k_grouped_fp8_gemm_tn_contiguous(a, sfa_words, b, sfb_words, ks, c=None,
                                     experts=None, rows=None):
    """a: uint8 [K_total, M] (MN-major); sfa_words: int32 [ceil(K_total/512)][align4(M)];
    b: uint8 [K_total, N]; sfb_words: int32 [ceil(K_total/512)][align4(N)];
    ks: per-expert K lengths (multiples of 128, summing to K_total);
    c: optional float32 [G, M, N].

    Returns {g: float64 [len(rows), N]} with D[g] = C[g] + A_g.T @ B_g, where A_g is
    rows [off_g, off_g + ks[g]) of A.  Scale of element (k, m): group k // 128 of
    column m, counted over the whole concatenated K axis."""
    k_total, m = a.shape
    n = b.shape[1]
    ks = [int(x) for x in ks]
    offs = np.concatenate([[0], np.cumsum(ks)]).astype(np.int64)
    assert offs[-1] == k_total
    rows = np.arange(m) if rows is None else np.asarray(rows)
    sa_all = row_scales(sfa_words, m, k_total)      # [M, K_total/128]
    sb_all = row_scales(sfb_words, n, k_total)      # [N, K_total/128]
    out = {}
    for e in (range(len(ks)) if experts is None else experts):
        lo, hi = offs[e], offs[e + 1]
        glo, ghi = lo // K_GROUP, hi // K_GROUP
        at = dequant_k_major(np.ascontiguousarray(a[lo:hi, rows].T), sa_all[rows, glo:ghi])
        bt = dequant_k_major(np.ascontiguousarray(b[lo:hi].T), sb_all[:, glo:ghi])
        d = at @ bt.T
        if c is not None:
            d = d + np.asarray(c[e], dtype=np.float64)[rows]
        out[e] = d
    return out
