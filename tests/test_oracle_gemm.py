"""Pins for the GEMM oracle: exact rational brute force on tiny shapes, closed forms
(identity, one-hot, integer-valued, scale identification), the hand-derived fixtures
of tests/golden/closed_forms.json, and segment logic.  The mutation test plants
plausible mistakes in a copy of the oracle (on the CPU) and checks that the pins
catch every one of them."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import formats as F
from oracle import gemm as G
import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def test_contiguous_rows_left_untouched_and_expert_routing():
    g = np.random.Generator(np.random.PCG64(21))
    m_indices = np.array([1] * 3 + [-1] * 125 + [0] * 128, dtype=np.int32)
    a = P.rand_codes(g, (256, 128))
    b = P.rand_codes(g, (2, 16, 128))
    sfa = P.rand_words(g, 256, 1)
    sfb = np.stack([P.rand_words(g, 1, 1) for _ in range(2)])
    d, written = oracle.m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, m_indices)
    assert written.sum() == 131
    dense1 = oracle.fp8_gemm_nt(a[:3], F.pack_ue8m0(F.unpack_ue8m0(sfa, 256, 1)[:3]), b[1], sfb[1])
    assert np.array_equal(d[:3], dense1)


def test_masked_zero_and_full_masks():
    g = np.random.Generator(np.random.PCG64(22))
    a = P.rand_codes(g, (2, 130, 128))
    b = P.rand_codes(g, (2, 8, 128))
    sfa = np.stack([P.rand_words(g, 130, 1) for _ in range(2)])
    sfb = np.stack([P.rand_words(g, 1, 1) for _ in range(2)])
    out = oracle.m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, [0, 130])
    assert out[0].shape == (0, 8) and out[1].shape == (130, 8)
    assert np.array_equal(out[1], oracle.fp8_gemm_nt(a[1], sfa[1], b[1], sfb[1]))


def test_k_grouped_equals_dense_on_one_segment():
    # one expert over the whole K: the TN GEMM equals the NT GEMM of the transposes
    g = np.random.Generator(np.random.PCG64(23))
    k, m, n = 256, 7, 9
    a = P.rand_codes(g, (k, m))
    b = P.rand_codes(g, (k, n))
    sa = g.integers(120, 135, (m, 2), dtype=np.uint8)
    sb = g.integers(120, 135, (n, 2), dtype=np.uint8)
    out = oracle.k_grouped_fp8_gemm_tn_contiguous(a, F.pack_ue8m0(sa), b, F.pack_ue8m0(sb), [k])
    # dense form needs block scales for B: use n <= 128 and per-row B scale equal across rows
    sb_blk = np.tile(sb[:1], (n, 1))
    out2 = oracle.k_grouped_fp8_gemm_tn_contiguous(a, F.pack_ue8m0(sa), b, F.pack_ue8m0(sb_blk), [k])
    dense = oracle.fp8_gemm_nt(np.ascontiguousarray(a.T), F.pack_ue8m0(sa),
                               np.ascontiguousarray(b.T), F.pack_ue8m0(sb[:1]))
    assert np.array_equal(out2[0], dense)
    assert out[0].shape == (m, n)


# ------------------------------------------------------------------ mutants
def _bias8_table():
    t = F.E4M3_TABLE.copy()
    t[np.isfinite(t)] /= 2
    return t


def _unsigned_table():
    return np.abs(F.E4M3_TABLE)


def _unpack_reversed(words, mn, groups):
    w = np.asarray(words).view(np.uint32)
    out = np.empty((mn, groups), dtype=np.uint8)
    for g in range(groups):
        out[:, g] = (w[g // 4, :mn] >> np.uint32(8 * (3 - g % 4))) & 0xFF
    return out


def _block_scales_mod(sfb_words, n, k):
    blk = F.unpack_ue8m0(sfb_words, (n + 127) // 128, k // 128)
    return blk[np.arange(n) % blk.shape[0]]


def _dequant_no_scale(q, sf):
    return F.e4m3_to_f64(q)


_orig_nt = G.fp8_gemm_nt
_orig_kg = G.k_grouped_fp8_gemm_tn_contiguous
_orig_contig = G.m_grouped_fp8_gemm_nt_contiguous


def _nt_drop_c(a, sfa, b, sfb, c=None, rows=None):
    return _orig_nt(a, sfa, b, sfb, None, rows)


def _nt_minus_c(a, sfa, b, sfb, c=None, rows=None):
    d = _orig_nt(a, sfa, b, sfb, None, rows)
    return d if c is None else d - np.asarray(c, np.float64)[rows if rows is not None else slice(None)]


def _kg_shifted_offsets(a, sfa, b, sfb, ks, c=None, experts=None, rows=None):
    ks = list(ks)
    return _orig_kg(a, sfa, b, sfb, ks[1:] + ks[:1], c, experts, rows)


def _contig_pad_as_expert0(a, sfa, b, sfb, m_indices, rows=None):
    return _orig_contig(a, sfa, b, sfb, np.maximum(m_indices, 0), rows)


def _row_scale_transposed(sfa_words, mn, k):
    s = F.unpack_ue8m0(sfa_words, mn, k // 128)
    return s[::-1]


def _nn_b_read_as_nt(a, sfa, b, sfb, c=None, rows=None):
    return _orig_nt(a, sfa, b, sfb, c, rows)


def _tt_a_read_as_nt(a, sfa, b, sfb, c=None, rows=None):
    return _orig_nt(a, sfa, b, sfb, c, rows)


def _tn_operands_swapped(a, sfa, b, sfb, c=None, rows=None):
    return _orig_nt(np.ascontiguousarray(b.T), sfa, np.ascontiguousarray(a.T), sfb, c, rows)


def _contig_nn_b_read_as_nt(a, sfa, b, sfb, m_indices, rows=None):
    return _orig_contig(a, sfa, b, sfb, m_indices, rows)


import oracle.swiglu as SW

_orig_silu = SW.silu


def _swiglu_halves_swapped(h):
    h = np.asarray(h, dtype=np.float64)
    i = h.shape[-1] // 2
    return _orig_silu(h[..., i:]) * h[..., :i]


def _sigmoid_not_silu(x):
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def _silu_sign_flipped(x):
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(x))


import oracle.mqa as MQ


def _mqa_no_relu(q, kv, kv_sf, weights, ks, ke, clean_logits=True, rows=None):
    s_len, heads, dim = q.shape
    t_len = kv.shape[0]
    rows = np.arange(s_len) if rows is None else np.asarray(rows)
    kvd = F.e4m3_to_f64(kv) * np.asarray(kv_sf, np.float64)[:, None]
    out = np.full((len(rows), t_len), -np.inf if clean_logits else np.nan)
    for r, i in enumerate(rows):
        lo, hi = max(int(ks[i]), 0), min(int(ke[i]), t_len)
        if hi > lo:
            out[r, lo:hi] = (F.e4m3_to_f64(q[i]) @ kvd[lo:hi].T).T @ np.asarray(weights[i], np.float64)
    return out


def _mqa_range_inclusive(q, kv, kv_sf, weights, ks, ke, clean_logits=True, rows=None):
    return _orig_mqa(q, kv, kv_sf, weights, ks, np.asarray(ke) + 1, clean_logits, rows)


def _mqa_scale_dropped(q, kv, kv_sf, weights, ks, ke, clean_logits=True, rows=None):
    return _orig_mqa(q, kv, np.ones_like(kv_sf), weights, ks, ke, clean_logits, rows)


_orig_mqa = MQ.fp8_mqa_logits

import oracle.fp4 as FP4


def _fp4_unpack_swapped(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p >> 4
    out[..., 1::2] = p & 0xF
    return out


def _fp4_scales_per_128(sfb_words, n, k):
    # one scale per 128-wide K-group (the FP8 activation granularity) instead of per 32
    s = F.unpack_ue8m0(sfb_words, n, k // 32)
    return np.repeat(s[:, 0::4], 4, axis=1)


def _e2m1_bias_2():
    return FP4.E2M1_TABLE / 2


def _e2m1_subnormal_one():
    t = FP4.E2M1_TABLE.copy()
    t[1], t[9] = 1.0, -1.0
    return t


def _fp4_scale_dropped(packed, sf_bytes):
    return FP4.e2m1_to_f64(FP4.unpack_fp4(packed))


MUTANTS = {
    "mqa_relu_dropped": [(MQ, "fp8_mqa_logits", lambda: _mqa_no_relu)],
    "mqa_range_end_inclusive": [(MQ, "fp8_mqa_logits", lambda: _mqa_range_inclusive)],
    "mqa_kv_scale_dropped": [(MQ, "fp8_mqa_logits", lambda: _mqa_scale_dropped)],
    "swiglu_halves_swapped": [(SW, "swiglu", lambda: _swiglu_halves_swapped)],
    "silu_is_sigmoid": [(SW, "silu", lambda: _sigmoid_not_silu)],
    "silu_sign_flipped": [(SW, "silu", lambda: _silu_sign_flipped)],
    "nn_b_not_transposed": [(G, "fp8_gemm_nn", lambda: _nn_b_read_as_nt)],
    "tt_a_not_transposed": [(G, "fp8_gemm_tt", lambda: _tt_a_read_as_nt)],
    "tn_operands_swapped": [(G, "fp8_gemm_tn", lambda: _tn_operands_swapped)],
    "contiguous_nn_b_not_transposed": [(G, "m_grouped_fp8_gemm_nn_contiguous", lambda: _contig_nn_b_read_as_nt)],
    "e4m3_bias_8": [(F, "E4M3_TABLE", _bias8_table)],
    "e4m3_sign_dropped": [(F, "E4M3_TABLE", _unsigned_table)],
    "scale_bytes_reversed": [(G, "unpack_ue8m0", lambda: _unpack_reversed)],
    "b_block_index_mod": [(G, "block_scales", lambda: _block_scales_mod)],
    "scale_dropped": [(G, "dequant_k_major", lambda: _dequant_no_scale)],
    "c_dropped": [(G, "fp8_gemm_nt", lambda: _nt_drop_c)],
    "c_sign_wrong": [(G, "fp8_gemm_nt", lambda: _nt_minus_c)],
    "k_offsets_shifted": [(G, "k_grouped_fp8_gemm_tn_contiguous", lambda: _kg_shifted_offsets)],
    "padding_rows_computed": [(G, "m_grouped_fp8_gemm_nt_contiguous", lambda: _contig_pad_as_expert0)],
    "row_scales_wrong_row": [(G, "row_scales", lambda: _row_scale_transposed)],
    "fp4_nibbles_swapped": [(FP4, "unpack_fp4", lambda: _fp4_unpack_swapped)],
    "fp4_scale_per_128": [(FP4, "mx_scales", lambda: _fp4_scales_per_128)],
    "e2m1_bias_2": [(FP4, "E2M1_TABLE", _e2m1_bias_2)],
    "e2m1_subnormal_is_one": [(FP4, "E2M1_TABLE", _e2m1_subnormal_one)],
    "fp4_scale_dropped": [(FP4, "dequant_mxfp4", lambda: _fp4_scale_dropped)],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    for mod, attr, make in MUTANTS[name]:
        monkeypatch.setattr(mod, attr, make())
        # the package re-exports the GEMM entry points
        if hasattr(oracle, attr):
            monkeypatch.setattr(oracle, attr, getattr(mod, attr))
    caught = []
    for check in P.ALL_CHECKS:
        try:
            check()
        except Exception:  # noqa: BLE001 - any failure counts as caught
            caught.append(check.__name__)
    assert caught, f"no pin detects mutant {name}"


def _exact_and_magnitude(terms_a, terms_b):
    """Exact sum of the products and the sum of their magnitudes."""
    tot, mag = Fraction(0), Fraction(0)
    for x, y in zip(terms_a, terms_b):
        p = x * y
        tot += p
        mag += abs(p)
    return tot, mag


def test_oracle_long_k_wide_range_exact():
    """The accumulation case of the FP8 GEMM (article "Deepseek AI Libera DeepGEMM",
    "Details and technical benefits": fine-grained scales with FP32 promotion so that long
    accumulations stay accurate): at K = 16384 with per-group magnitudes spanning about
    +-20 binades, the oracle's FP64 result agrees with an exact rational sum over every
    term to FP64 rounding of the sum of magnitudes."""
    import workloads
    m, n, k = 3, 130, 16384
    w = workloads.dense_wide_range(77, m, n, k, True)
    a, sa = F.quantize_rows(w["a"])
    b, sb = F.quantize_blocks(w["b"])
    sfa, sfb = F.pack_ue8m0(sa), F.pack_ue8m0(sb)
    got = oracle.fp8_gemm_nt(a, sfa, b, sfb, w["c"])
    # the scales really span the intended range (bytes 127 +- about 10 each)
    assert int(sa.max()) - int(sa.min()) >= 18 and int(sb.max()) - int(sb.min()) >= 18
    for (i, j) in [(0, 0), (1, 129), (2, 64)]:
        ta = [P.fr_e4m3(a[i, kk]) * P.fr_ue8(P.word_byte(sfa, kk // 128, i)) for kk in range(k)]
        tb = [P.fr_e4m3(b[j, kk]) * P.fr_ue8(P.word_byte(sfb, kk // 128, j // 128)) for kk in range(k)]
        tot, mag = _exact_and_magnitude(ta, tb)
        tot += Fraction(float(w["c"][i, j]))
        assert P.close_fp64(float(got[i, j]), tot, mag + 1, k), (i, j)
        # the falling magnitudes: the last quarter of K contributes far less than the first
        q = k // 4
        first, _ = _exact_and_magnitude(ta[:q], tb[:q])
        _, last_mag = _exact_and_magnitude(ta[-q:], tb[-q:])
        assert last_mag < Fraction(1, 2 ** 10) * max(abs(first), Fraction(1, 2 ** 20))


def test_oracle_k_grouped_single_long_segment_exact():
    """One expert owns the whole K axis (ks = [16384, 0, 0]): its output is the exact
    rational sum; the empty experts' outputs are C."""
    import workloads
    m, n = 2, 3
    w = workloads.k_grouped_wide_range(78, [16384, 0, 0], m, n)
    a, sa = F.quantize_cols(w["a"])
    b, sb = F.quantize_cols(w["b"])
    sfa, sfb = F.pack_ue8m0(sa), F.pack_ue8m0(sb)
    out = oracle.k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, w["ks"], w["c"])
    for (i, j) in [(0, 0), (1, 2)]:
        exact = P.exact_k_grouped(a, sfa, b, sfb, w["ks"], w["c"], 0, i, j)
        ta = [P.fr_e4m3(a[kk, i]) * P.fr_ue8(P.word_byte(sfa, kk // 128, i)) for kk in range(16384)]
        tb = [P.fr_e4m3(b[kk, j]) * P.fr_ue8(P.word_byte(sfb, kk // 128, j)) for kk in range(16384)]
        _, mag = _exact_and_magnitude(ta, tb)
        assert P.close_fp64(float(out[0][i, j]), exact, mag + 1, 16384), (i, j)
    for e in (1, 2):
        assert np.array_equal(out[e], w["c"][e].astype(np.float64))
