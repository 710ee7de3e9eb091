"""SwiGLU + per-1x128 FP8 requantisation after the gate-up GEMM, as plain FP64 definitions.

TEST INFRASTRUCTURE (oracle): see the header of ``oracle/formats.py`` for who may
import it.  Shares no code with the CUDA library.

What is computed.  The MoE MLP runs linear 1 (gate and up projections), SwiGLU, then
linear 2 (the down projection) whose FP8 A operand is the SwiGLU output re-quantised
per token and 128-channel group ("Mega MoE", docsearch / README; the staged path's
"K2: SwiGLU + channelwise FP8 quant", MegaMoE DCU README "Runtime Routing").  Readings
where the pages are silent (stated in the design notes): the gate-up weight of each
expert is [2I, K] with the I gate rows first and the I up rows after them, so the GEMM
output row h = [gate | up]; SwiGLU(h)[i] = SiLU(gate[i]) * up[i] with
SiLU(x) = x / (1 + exp(-x)); the result is quantised like any activation: per row and
1x128 group along I, scale 2^e with the smallest e such that amax <= 448 * 2^e, codes
E4M3 round-to-nearest-even.  The quantisation decision is taken on FP32 values (the
precision of the kernel's epilogue): the FP64 SwiGLU value is rounded to FP32 first.
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from .gemm import m_grouped_fp8_gemm_nt_contiguous, m_grouped_fp8_gemm_nt_masked


def silu(x) -> np.ndarray:
    """SiLU (swish) in FP64: x / (1 + exp(-x)); exp overflow for very negative x gives -0."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def swiglu(h) -> np.ndarray:
    """h[..., 2I] = [gate | up] -> SiLU(gate) * up, shape [..., I]."""
    h = np.asarray(h, dtype=np.float64)
    i = h.shape[-1] // 2
    return silu(h[..., :i]) * h[..., i:]


def swiglu_quantize(h):
    """[R, 2I] FP64 GEMM output -> (codes uint8 [R, I], scale bytes uint8 [R, I/128])."""
    y32 = swiglu(h).astype(np.float32)
    return F.quantize_rows(y32.astype(np.float64))


def m_grouped_fp8_gemm_nt_contiguous_swiglu(a, sfa_words, b, sfb_words, m_indices, rows=None):
    """Gate-up GEMM of the contiguous layout (b [G, 2I, K]) followed by SwiGLU and the
    per-1x128 requantisation.  Returns (codes [len(rows), I], scale bytes
    [len(rows), I/128], written bool [len(rows)]); padding rows (-1) are not written
    (their codes are 0 and scale bytes 0 here)."""
    h, written = m_grouped_fp8_gemm_nt_contiguous(a, sfa_words, b, sfb_words, m_indices, rows)
    i = b.shape[1] // 2
    q = np.zeros((h.shape[0], i), np.uint8)
    sf = np.zeros((h.shape[0], i // F.K_GROUP), np.uint8)
    if written.any():
        q[written], sf[written] = swiglu_quantize(h[written])
    return q, sf, written


def m_grouped_fp8_gemm_nt_masked_swiglu(a, sfa_words, b, sfb_words, masked_m, experts=None):
    """Gate-up GEMM of the masked layout followed by SwiGLU and the per-1x128
    requantisation: {g: (codes [masked_m[g], I], scale bytes [masked_m[g], I/128])}."""
    d = m_grouped_fp8_gemm_nt_masked(a, sfa_words, b, sfb_words, masked_m, experts)
    out = {}
    for g, h in d.items():
        i = b.shape[1] // 2
        if h.shape[0] == 0:
            out[g] = (np.zeros((0, i), np.uint8), np.zeros((0, i // F.K_GROUP), np.uint8))
        else:
            out[g] = swiglu_quantize(h)
    return out
