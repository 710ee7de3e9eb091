"""Number formats and layouts of the fine-grained FP8 GEMM, written out plainly.

TEST INFRASTRUCTURE (oracle). Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this package.
The CUDA library never imports, links or calls it, and it shares no code with the
CUDA library.

Sources, by page and section:

* "DeepGEMM Documentation" (docsearch index), section 4 "Understand DeepGEMM GEMM
  Naming and Layouts", and the yuguo-Jack/DeepGEMM README, "Interfaces > Notices":
  SM100 takes scaling factors as packed UE8M0, four UE8M0 values in one 32-bit
  ``torch.int``; the LHS scaling factors are TMA-aligned and transposed (MN-major).
  The Chinese post (bittide, section "接口 / 注意事项") links the PTX ISA section
  "alternate floating point data formats" for UE8M0.
* Same sections: the user does the FP8 cast; the library's packing helpers are
  ``get_tma_aligned_size`` and ``get_mn_major_tma_aligned_packed_ue8m0_tensor``
  (docsearch section 10, README "Utilities").

Readings taken where the pages are silent:

* E4M3 is the OCP FP8 "fn" variant: bias 7, no infinities, S.1111.111 is NaN,
  largest finite 448.
* Byte j (bits 8j..8j+7) of packed word w holds the scale of K-group 4w+j.
* The packed array is [ceil(groups/4)][align4(MN)] int32: MN padded to a multiple of
  4 words (16 bytes, the TMA stride rule); padding words are zero and ignored.
* Quantiser (used only to make inputs): per group, the scale is the smallest power of
  two s with amax/s <= 448; the code is E4M3 round-to-nearest-even of x/s.
* Output rounding: BF16 round-to-nearest-even of the exact (FP64) result; FP32
  round-to-nearest-even.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
K_GROUP = 128          # one scale per 128 consecutive K elements
PACK = 4               # UE8M0 bytes per packed int32 word
TMA_ALIGN_BYTES = 16   # TMA requires 16-byte aligned strides


# ---------------------------------------------------------------------------
# E4M3
# ---------------------------------------------------------------------------
def e4m3_value(code: int) -> float:
    """Value of one E4M3 byte from its bit fields: sign s, exponent e (4 bits,
    bias 7), mantissa m (3 bits).  e == 0 is subnormal: (m/8) * 2^-6.  Otherwise
    (1 + m/8) * 2^(e-7).  e == 15 with m == 7 is NaN; there is no infinity."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E4M3_TABLE.setflags(write=False)


def e4m3_to_f64(q) -> np.ndarray:
    """Exact decode of an array of E4M3 bytes to float64."""
    return E4M3_TABLE[np.asarray(q, dtype=np.uint8)]


def f64_to_e4m3(x) -> np.ndarray:
    """E4M3 round-to-nearest-even of float64 values (returns the bytes).

    Normal range (|x| >= 2^-6): the spacing of representable values at exponent
    e = floor(log2|x|) is 2^(e-3); subnormal range: spacing 2^-9.  The value is
    rounded to a multiple of the spacing with ties to even (np.rint), clamped to
    +-448 (saturation; never reached by the quantiser, whose inputs satisfy
    |x| <= 448), and then re-encoded from its exponent and mantissa.  NaN encodes
    as 0x7F.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                     # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)              # exponent of the leading bit, subnormals share -6
    spacing = np.ldexp(1.0, e - 3)
    r = np.rint(a / spacing) * spacing      # exact: division by a power of two
    r = np.minimum(r, E4M3_MAX)
    # re-encode the rounded magnitude
    _, rex = np.frexp(r)
    re = rex - 1
    normal = r >= 2.0 ** -6
    exp_field = np.where(normal, re + 7, 0)
    man_field = np.where(normal,
                         np.rint((r / np.ldexp(1.0, np.where(normal, re, 0)) - 1.0) * 8.0),
                         np.rint(r / 2.0 ** -9))
    code = (exp_field.astype(np.int64) << 3) | man_field.astype(np.int64)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


# ---------------------------------------------------------------------------
# UE8M0
# ---------------------------------------------------------------------------
def ue8m0_to_f64(u) -> np.ndarray:
    """UE8M0: an unsigned 8-bit exponent, value 2^(u-127); u == 255 is NaN."""
    u = np.asarray(u, dtype=np.uint8).astype(np.int64)
    out = np.ldexp(1.0, u - 127)
    return np.where(u == 255, np.nan, out)


def ue8m0_for_amax(amax) -> np.ndarray:
    """Scale byte for a group whose largest magnitude is ``amax``: the smallest
    power of two 2^e with amax <= 448 * 2^e, as the byte e + 127 (clamped to
    [0, 254]).  amax == 0 gives 127 (scale 1).  The estimate from log2 is fixed up
    with exact comparisons, so the result is exact for every float input."""
    amax = np.asarray(amax, dtype=np.float64)
    safe = np.where(amax > 0, amax, 1.0)
    e = np.ceil(np.log2(safe / E4M3_MAX)).astype(np.int64)
    # exact fix-up: want amax <= 448*2^e and amax > 448*2^(e-1)
    too_small = safe > E4M3_MAX * np.ldexp(1.0, e)
    e = np.where(too_small, e + 1, e)
    too_big = safe <= E4M3_MAX * np.ldexp(1.0, e - 1)
    e = np.where(too_big, e - 1, e)
    byte = np.clip(e + 127, 0, 254)
    byte = np.where(amax > 0, byte, 127)
    return byte.astype(np.uint8)


# ---------------------------------------------------------------------------
# BF16 / FP32 output rounding
# ---------------------------------------------------------------------------
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def f64_to_bf16(x) -> np.ndarray:
    """BF16 round-to-nearest-even of float64 values; returns the 16-bit patterns.

    BF16 has 8 significant bits: at exponent e (clamped to -126 below the normal
    range) the spacing is 2^(e-7).  Magnitudes that round above the largest finite
    BF16 become infinity."""
    x = np.asarray(x, dtype=np.float64)
    _, ex = np.frexp(x)
    e = np.maximum(ex - 1, -126)
    spacing = np.ldexp(1.0, e - 7)
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.rint(x / spacing) * spacing
        r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, x), r)
    r = np.where(np.isfinite(x), r, x)
    bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return np.where(np.isnan(x), np.uint16(0x7FC0), bits).astype(np.uint16)


def bf16_to_f64(bits) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def f64_to_f32(x) -> np.ndarray:
    """FP32 round-to-nearest-even (numpy's conversion)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


# ---------------------------------------------------------------------------
# Packed, MN-major, TMA-aligned scale layout
# ---------------------------------------------------------------------------
def tma_aligned_size(x: int, elem_bytes: int) -> int:
    """Round x up so that x * elem_bytes is a multiple of 16 bytes
    (``get_tma_aligned_size``, docsearch section 10)."""
    per = TMA_ALIGN_BYTES // elem_bytes
    return (x + per - 1) // per * per


def pack_ue8m0(sf: np.ndarray) -> np.ndarray:
    """Pack scale bytes sf[MN, groups] into int32 words [ceil(groups/4)][align4(MN)].

    Word w of row i holds groups 4w..4w+3 of that row, byte j (bits 8j..8j+7) being
    group 4w+j.  Missing tail groups and padding rows are zero."""
    sf = np.asarray(sf, dtype=np.uint8)
    mn, groups = sf.shape
    words = np.zeros(((groups + PACK - 1) // PACK, tma_aligned_size(mn, 4)), dtype=np.uint32)
    for g in range(groups):
        words[g // PACK, :mn] |= sf[:, g].astype(np.uint32) << np.uint32(8 * (g % PACK))
    return words.view(np.int32)


def unpack_ue8m0(words: np.ndarray, mn: int, groups: int) -> np.ndarray:
    """Inverse of :func:`pack_ue8m0`: scale bytes [mn, groups]."""
    w = np.asarray(words).view(np.uint32)
    out = np.empty((mn, groups), dtype=np.uint8)
    for g in range(groups):
        out[:, g] = (w[g // PACK, :mn] >> np.uint32(8 * (g % PACK))) & 0xFF
    return out


# ---------------------------------------------------------------------------
# Quantisers (input preparation; the GEMM consumes their bytes)
# ---------------------------------------------------------------------------
def quantize_rows(x: np.ndarray):
    """Per 1x128 group along the last axis: x[R, K] -> (codes uint8[R, K],
    scale bytes uint8[R, K/128]).  K must be a multiple of 128."""
    x = np.asarray(x, dtype=np.float64)
    r, k = x.shape
    assert k % K_GROUP == 0
    g = x.reshape(r, k // K_GROUP, K_GROUP)
    sf = ue8m0_for_amax(np.abs(g).max(axis=2))
    s = ue8m0_to_f64(sf)[:, :, None]
    q = f64_to_e4m3(g / s).reshape(r, k)
    return q, sf


def quantize_blocks(w: np.ndarray):
    """Per 128x128 block: w[N, K] -> (codes uint8[N, K], scale bytes
    uint8[ceil(N/128), K/128]).  A ragged last row-block uses its valid rows."""
    w = np.asarray(w, dtype=np.float64)
    n, k = w.shape
    assert k % K_GROUP == 0
    nb = (n + K_GROUP - 1) // K_GROUP
    q = np.empty((n, k), dtype=np.uint8)
    sf = np.empty((nb, k // K_GROUP), dtype=np.uint8)
    for i in range(nb):
        blk = w[i * K_GROUP:(i + 1) * K_GROUP].reshape(-1, k // K_GROUP, K_GROUP)
        sf[i] = ue8m0_for_amax(np.abs(blk).max(axis=(0, 2)))
        s = ue8m0_to_f64(sf[i])[None, :, None]
        q[i * K_GROUP:(i + 1) * K_GROUP] = f64_to_e4m3(blk / s).reshape(-1, k)
    return q, sf


def quantize_cols(x: np.ndarray):
    """Per 1x128 group along the FIRST axis (MN-major operands of the K-grouped
    GEMM): x[K, MN] -> (codes uint8[K, MN], scale bytes uint8[MN, K/128])."""
    q_t, sf = quantize_rows(np.asarray(x).T)
    return np.ascontiguousarray(q_t.T), sf


def ceil_div(a: int, b: int) -> int:
    return (a + b - 1) // b


def log2_exact(x: float) -> int:
    """Exponent of an exact power of two (used by tests)."""
    m, e = math.frexp(x)
    assert m == 0.5
    return e - 1
