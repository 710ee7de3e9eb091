"""Pins for the oracle's number formats, quantiser and scale packing.

Each check compares the oracle with something other than itself: PyTorch's own
FP8 / E8M0 / BF16 conversions (library routines), exact rational arithmetic, and the
hand-derived fixtures in tests/golden/closed_forms.json."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))


def _same(x, y):
    x, y = np.asarray(x, np.float64), np.asarray(y, np.float64)
    return np.array_equal(np.isnan(x), np.isnan(y)) and np.array_equal(
        np.nan_to_num(x, nan=0.0), np.nan_to_num(y, nan=0.0)) and np.array_equal(
        np.signbit(np.nan_to_num(x)), np.signbit(np.nan_to_num(y)))


# --------------------------------------------------------------------- E4M3
def test_e4m3_table_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    assert _same(F.E4M3_TABLE, ref)


def test_e4m3_landmarks():
    for row in GOLDEN["e4m3"]:
        got = F.e4m3_to_f64(np.array([int(row["code"], 16)]))[0]
        want = float("nan") if row["value"] == "nan" else row["value"]
        assert _same([got], [want]), row


def test_e4m3_table_from_bits_with_fractions():
    # independent evaluation of every code with exact rationals
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            assert math.isnan(F.E4M3_TABLE[code])
            continue
        mag = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        assert Fraction(F.E4M3_TABLE[code]) == (-mag if s else mag)


def test_e4m3_encode_matches_torch_random_and_ties():
    g = np.random.Generator(np.random.PCG64(7))
    x = np.concatenate([
        g.standard_normal(200_000) * 60,
        g.standard_normal(50_000) * 0.01,          # subnormal region
        g.uniform(-448, 448, 50_000),
    ])
    pos = F.E4M3_TABLE[:127]
    mids = (pos[:-1] + pos[1:]) / 2                # exact ties between neighbours
    x = np.concatenate([x, mids, -mids, pos, -pos, [0.0, -0.0, 448.0, -448.0]])
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.f64_to_e4m3(x)
    assert np.array_equal(got, ref)


def test_e4m3_encode_round_trip_every_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(F.f64_to_e4m3(F.e4m3_to_f64(codes)), codes)


# -------------------------------------------------------------------- UE8M0
def test_ue8m0_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = F.ue8m0_to_f64(np.arange(256))
    assert _same(got, ref)


def test_ue8m0_landmarks():
    for row in GOLDEN["ue8m0"]:
        got = F.ue8m0_to_f64(np.array([row["code"]]))[0]
        want = float("nan") if row["value"] == "nan" else row["value"]
        assert _same([got], [want]), row


def test_power_of_two_scaling_is_exact():
    # dec8(q) * 2^s is exact in FP64 for all finite codes and s in [-127, 127]
    vals = F.E4M3_TABLE[np.isfinite(F.E4M3_TABLE)]
    for s in range(-127, 128):
        prod = vals * F.ue8m0_to_f64(np.array([s + 127]))[0]
        for v, p in zip(vals[::7], prod[::7]):
            assert Fraction(p) == Fraction(v) * Fraction(2) ** s


# --------------------------------------------------------------------- BF16
def test_bf16_matches_torch():
    g = np.random.Generator(np.random.PCG64(3))
    x32 = np.concatenate([
        g.standard_normal(300_000).astype(np.float32) * np.float32(1e3),
        (g.standard_normal(20_000) * 1e-39).astype(np.float32),    # subnormal
        np.array([3.38e38, -3.39e38, 1e-45, 0.0, -0.0], dtype=np.float32),
    ])
    # exact ties: bf16 value + half a bf16 spacing (representable in fp32)
    base = torch.from_numpy(x32[:1000]).to(torch.bfloat16).to(torch.float32).numpy()
    _, ex = np.frexp(base.astype(np.float64))
    ties = (base.astype(np.float64) + np.ldexp(1.0, ex - 1 - 8)).astype(np.float32)
    x32 = np.concatenate([x32, ties])
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = F.f64_to_bf16(x32.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_overflow_and_nan():
    got = F.f64_to_bf16(np.array([1e39, -1e39, np.inf, np.nan]))
    assert list(got[:3]) == [0x7F80, 0xFF80, 0x7F80] and got[3] == 0x7FC0


# ---------------------------------------------------------------- quantiser
def test_scale_choice_is_smallest_power_of_two():
    g = np.random.Generator(np.random.PCG64(11))
    amax = np.concatenate([np.abs(g.standard_normal(20000)) * 10 ** g.uniform(-8, 8, 20000),
                           [448.0, 448.0 * 2 ** 5, 448.0 * 2 ** -3, 1e-30, 0.0]])
    byte = F.ue8m0_for_amax(amax)
    for a, b in zip(amax, byte):
        if a == 0:
            assert b == 127
            continue
        e = int(b) - 127
        # exact rationals: a <= 448 * 2^e and a > 448 * 2^(e-1)
        assert Fraction(a) <= 448 * Fraction(2) ** e
        assert Fraction(a) > 448 * Fraction(2) ** (e - 1)


def test_quantize_rows_against_brute_force():
    g = np.random.Generator(np.random.PCG64(5))
    x = (g.standard_normal((3, 256)) * 3).astype(np.float32)
    q, sf = F.quantize_rows(x)
    for r in range(3):
        for grp in range(2):
            seg = x[r, grp * 128:(grp + 1) * 128].astype(np.float64)
            s = Fraction(2) ** (int(sf[r, grp]) - 127)
            assert max(abs(Fraction(v)) for v in seg) / s <= 448
            finite = [Fraction(v) for v in F.E4M3_TABLE if np.isfinite(v)]
            for j in range(0, 128, 9):
                t = Fraction(seg[j]) / s
                best = min(abs(t - f) for f in finite)
                assert abs(Fraction(F.e4m3_to_f64([q[r, grp * 128 + j]])[0]) - t) == best


def test_quantize_blocks_shares_one_scale_per_128x128():
    g = np.random.Generator(np.random.PCG64(6))
    w = g.standard_normal((200, 256)).astype(np.float32)
    w[130, 5] = 1000.0
    q, sf = F.quantize_blocks(w)
    assert sf.shape == (2, 2)
    # block (1, 0) holds the outlier; its scale must cover it
    assert F.ue8m0_to_f64(sf[1, 0]) * 448 >= 1000.0 > F.ue8m0_to_f64(sf[1, 0]) * 224
    assert F.e4m3_to_f64(q[130, 5]) * F.ue8m0_to_f64(sf[1, 0]) == pytest.approx(1000.0, rel=1 / 16)


def test_quantize_cols_is_rows_transposed():
    g = np.random.Generator(np.random.PCG64(8))
    x = g.standard_normal((256, 40)).astype(np.float32)
    q, sf = F.quantize_cols(x)
    qr, sfr = F.quantize_rows(x.T)
    assert np.array_equal(q, qr.T) and np.array_equal(sf, sfr)


# ------------------------------------------------------------------ packing
def test_pack_golden():
    p = GOLDEN["packing"]
    words = F.pack_ue8m0(np.array(p["sf_rows"], dtype=np.uint8))
    want = np.array([[int(v, 16) for v in row] for row in p["words_hex"]], dtype=np.uint32)
    assert np.array_equal(words.view(np.uint32), want)


def test_pack_round_trip_and_alignment():
    g = np.random.Generator(np.random.PCG64(9))
    for mn, groups in [(1, 1), (5, 3), (128, 16), (130, 33)]:
        sf = g.integers(0, 256, (mn, groups), dtype=np.uint8)
        w = F.pack_ue8m0(sf)
        assert w.dtype == np.int32 and w.shape == (math.ceil(groups / 4), F.tma_aligned_size(mn, 4))
        assert (w.shape[1] * 4) % 16 == 0
        assert np.array_equal(F.unpack_ue8m0(w, mn, groups), sf)
        assert np.all(w[:, mn:] == 0)


def test_tma_aligned_size():
    assert [F.tma_aligned_size(x, 4) for x in (0, 1, 4, 5, 64, 65)] == [0, 4, 4, 8, 64, 68]
    assert [F.tma_aligned_size(x, 1) for x in (1, 16, 17)] == [16, 16, 32]
