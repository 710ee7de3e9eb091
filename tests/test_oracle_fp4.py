"""Pins for the FP8 x FP4 oracle's number formats and quantiser.

Checked against something other than the oracle itself: exact rationals from the E2M1 bit
fields, the E4M3 table (every E2M1 value must be an E4M3 value, since both are minifloats
with at least E2M1's exponent range and mantissa), brute-force nearest-value search for the
quantiser, and the MX scale rule (6 * 2^(e-1) < amax <= 6 * 2^e).  The FP4 GEMM itself is
pinned by the exact brute force and golden cases in ``oracle_pins.py`` (run by
``test_oracle_gemm.py``, which also plants mistakes in the FP4 oracle)."""
from fractions import Fraction

import numpy as np

from oracle import formats as F
from oracle import fp4
import oracle_pins as P


def test_e2m1_table_from_bits_with_fractions():
    for code in range(16):
        assert Fraction(fp4.E2M1_TABLE[code]) == P.fr_e2m1(code), code


def test_e2m1_values_are_e4m3_values():
    e4m3 = set(F.E4M3_TABLE[np.isfinite(F.E4M3_TABLE)].tolist())
    assert set(fp4.E2M1_TABLE.tolist()) <= e4m3
    assert sorted(set(np.abs(fp4.E2M1_TABLE).tolist())) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _nearest_even(x: float) -> int:
    """Brute force: the non-negative code nearest |x| (ties to the code with mantissa bit
    0), magnitudes above 6 clamped, sign bit from x."""
    best = None
    for code in range(8):
        d = abs(abs(x) - float(P.fr_e2m1(code)))
        key = (d, code & 1)
        if best is None or key < best[0]:
            best = (key, code)
    code = 7 if abs(x) > 6 else best[1]
    return code | (8 if np.signbit(x) else 0)


def test_e2m1_rounding_brute_force_with_every_tie():
    g = np.random.Generator(np.random.PCG64(31))
    mags = np.array(sorted(set(np.abs(fp4.E2M1_TABLE).tolist())))
    ties = (mags[:-1] + mags[1:]) / 2
    x = np.concatenate([g.uniform(-8, 8, 4000), ties, -ties, mags, -mags, [6.5, -7.0, 1e9]])
    got = fp4.f64_to_e2m1(x)
    for xi, ci in zip(x, got):
        assert int(ci) == _nearest_even(float(xi)), (xi, ci)


def test_pack_unpack_round_trip_and_nibble_order():
    g = np.random.Generator(np.random.PCG64(32))
    codes = g.integers(0, 16, (5, 64), dtype=np.uint8)
    packed = fp4.pack_fp4(codes)
    assert packed.shape == (5, 32)
    assert np.array_equal(fp4.unpack_fp4(packed), codes)
    for kk in range(64):
        assert np.all([P.fp4_code(packed[r], kk) == codes[r, kk] for r in range(5)])


def test_mx_quantiser_scale_rule_and_error_bound():
    g = np.random.Generator(np.random.PCG64(33))
    w = g.standard_normal((6, 256)) * np.exp2(g.integers(-20, 20, (6, 1)))
    w[0, :32] = 0.0                                       # an all-zero block
    packed, sf = fp4.quantize_mxfp4(w)
    assert packed.shape == (6, 128) and sf.shape == (6, 8)
    assert sf[0, 0] == 127
    amax = np.abs(w.reshape(6, 8, 32)).max(axis=2)
    s = np.exp2(sf.astype(np.float64) - 127)
    nz = amax > 0
    assert np.all(amax[nz] <= 6 * s[nz]) and np.all(amax[nz] > 3 * s[nz])
    deq = fp4.dequant_mxfp4(packed, sf)
    # RNE within each block: half a spacing, the largest spacing being 2 * s
    assert np.all(np.abs(deq - w) <= np.repeat(s, 32, axis=1) + 1e-300)
    # codes decode to the nearest E2M1 value of w / s
    q = fp4.unpack_fp4(packed)
    scaled = w / np.repeat(s, 32, axis=1)
    for r in range(6):
        for kk in range(0, 256, 7):
            assert int(q[r, kk]) & 7 == _nearest_even(float(scaled[r, kk])) & 7


def test_mx_scale_packing_is_the_fp8_packing_at_32_wide_blocks():
    # four 32-blocks a word, one word per 128-wide K-group: byte j of word w is block 4w + j
    sf = np.arange(24, dtype=np.uint8).reshape(3, 8) + 100
    words = fp4.pack_mx_scales(sf)
    assert words.shape == (2, 4)
    for r in range(3):
        for blk in range(8):
            assert P.word_byte(words, blk, r) == sf[r, blk]
