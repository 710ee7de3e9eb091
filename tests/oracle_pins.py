"""Pin checks for the GEMM oracle, written as plain functions so that the tests can
run them on the oracle as it is and on deliberately broken copies of it (a pin that
cannot tell a broken oracle from the real one pins nothing).

The independent evaluator here works element by element with exact rationals
(``fractions.Fraction``), decodes E4M3 and UE8M0 from their bit fields and reads the
packed scale words with integer shifts.  It shares no code with ``oracle/``."""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))


# ------------------------------------------------------------- exact decode
def fr_e4m3(code: int) -> Fraction:
    code = int(code)
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    assert not (e == 15 and m == 7), "NaN code in brute-force input"
    mag = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -mag if s else mag


def fr_ue8(byte: int) -> Fraction:
    assert byte != 255
    return Fraction(2) ** (int(byte) - 127)


def word_byte(words: np.ndarray, group: int, index: int) -> int:
    w = int(np.asarray(words).view(np.uint32)[group // 4, index])
    return (w >> (8 * (group % 4))) & 0xFF


def fr_to_bf16_bits(x: Fraction) -> int:
    """Exact round-to-nearest-even of a rational to BF16 bits (finite range only)."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    q = a / Fraction(2) ** (e - 7)
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = fl * Fraction(2) ** (e - 7)
    f32 = np.float32(float(val))          # exactly representable
    return sign | int(np.array([f32]).view(np.uint32)[0] >> 16)


# -------------------------------------------------------- exact references
def exact_dense(a, sfa, b, sfb, c, m, n) -> Fraction:
    k = a.shape[1]
    tot = Fraction(0) if c is None else Fraction(float(c[m, n]))
    for kk in range(k):
        g = kk // 128
        tot += (fr_e4m3(a[m, kk]) * fr_ue8(word_byte(sfa, g, m)) *
                fr_e4m3(b[n, kk]) * fr_ue8(word_byte(sfb, g, n // 128)))
    return tot


def exact_layout(a, sfa, b, sfb, c, m, n, a_t, b_n) -> Fraction:
    """Element (m, n) with A stored [K][M] when a_t (else [M][K]) and B stored [K][N]
    when b_n (else [N][K]); scales in the NT layouts."""
    k = a.shape[0] if a_t else a.shape[1]
    tot = Fraction(0) if c is None else Fraction(float(c[m, n]))
    for kk in range(k):
        g = kk // 128
        av = a[kk, m] if a_t else a[m, kk]
        bv = b[kk, n] if b_n else b[n, kk]
        tot += fr_e4m3(av) * fr_ue8(word_byte(sfa, g, m)) * fr_e4m3(bv) * fr_ue8(word_byte(sfb, g, n // 128))
    return tot


def exact_k_grouped(a, sfa, b, sfb, ks, c, e, m, n) -> Fraction:
    off = int(sum(ks[:e]))
    tot = Fraction(0) if c is None else Fraction(float(c[e, m, n]))
    for kk in range(off, off + int(ks[e])):
        g = kk // 128
        tot += (fr_e4m3(a[kk, m]) * fr_ue8(word_byte(sfa, g, m)) *
                fr_e4m3(b[kk, n]) * fr_ue8(word_byte(sfb, g, n)))
    return tot


# ------------------------------------------------------------ input makers
def rand_codes(g, shape):
    q = g.integers(0, 256, shape, dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38        # no NaN in valid data
    return q


def rand_words(g, mn, groups, lo=118, hi=137):
    from oracle.formats import pack_ue8m0   # packing is pinned by its own golden test
    return pack_ue8m0(g.integers(lo, hi, (mn, groups), dtype=np.uint8))


def close_fp64(got: float, exact: Fraction, mag: Fraction, k: int) -> bool:
    return abs(Fraction(got) - exact) <= mag * k * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 1000)


# ------------------------------------------------------------------- checks
def check_golden_gemm():
    import oracle
    from oracle.formats import pack_ue8m0
    for case in GOLDEN["gemm_nt"]:
        m, n, k = case["M"], case["N"], case["K"]
        a = np.full((m, k), int(case["a"], 16), np.uint8)
        b = np.full((n, k), int(case["b"], 16), np.uint8)
        sfa = pack_ue8m0(np.tile(np.array(case["sa"], np.uint8), (m, 1)))
        sfb = pack_ue8m0(np.tile(np.array(case["sb"], np.uint8), ((n + 127) // 128, 1)))
        c = None if case["c"] is None else np.full((m, n), case["c"], np.float32)
        d = oracle.fp8_gemm_nt(a, sfa, b, sfb, c)
        assert np.all(d == case["expect"]), (case["name"], d)


def check_dense_brute_force(seed=0):
    import oracle
    g = np.random.Generator(np.random.PCG64(seed))
    for (m, n, k, with_c) in [(3, 5, 128, False), (2, 131, 384, True), (4, 7, 640, False)]:
        a, b = rand_codes(g, (m, k)), rand_codes(g, (n, k))
        sfa, sfb = rand_words(g, m, k // 128), rand_words(g, (n + 127) // 128, k // 128)
        c = g.standard_normal((m, n)).astype(np.float32) if with_c else None
        d = oracle.fp8_gemm_nt(a, sfa, b, sfb, c)
        bits = oracle.round_output(d, "bf16")
        cols = range(n) if n < 16 else [0, 1, 64, 127, 128, 129, 130]
        for i in range(m):
            for j in cols:
                ex = exact_dense(a, sfa, b, sfb, c, i, j)
                mag = sum(abs(fr_e4m3(a[i, kk]) * fr_e4m3(b[j, kk])) for kk in range(k)) * Fraction(2) ** 40
                assert close_fp64(d[i, j], ex, mag, k), (m, n, k, i, j)
                assert bits[i, j] == fr_to_bf16_bits(ex), (i, j)


def check_layouts_brute_force(seed=5):
    """NN, TN, TT against the exact sum read straight from the stored arrays; the square
    case makes a transposition mistake silent in shape, so only the values can tell."""
    import oracle
    g = np.random.Generator(np.random.PCG64(seed))
    fns = {"nn": (oracle.fp8_gemm_nn, False, True), "tn": (oracle.fp8_gemm_tn, True, True),
           "tt": (oracle.fp8_gemm_tt, True, False)}
    for name, (fn, a_t, b_n) in fns.items():
        for (m, n, k, with_c) in [(128, 128, 128, False), (3, 130, 256, True)]:
            a = rand_codes(g, (k, m) if a_t else (m, k))
            b = rand_codes(g, (k, n) if b_n else (n, k))
            sfa, sfb = rand_words(g, m, k // 128), rand_words(g, (n + 127) // 128, k // 128)
            c = g.standard_normal((m, n)).astype(np.float32) if with_c else None
            d = fn(a, sfa, b, sfb, c)
            assert d.shape == (m, n), name
            for i in (0, 1, m - 1):
                for j in (0, 2, n - 1):
                    ex = exact_layout(a, sfa, b, sfb, c, i, j, a_t, b_n)
                    assert abs(Fraction(d[i, j]) - ex) <= (abs(ex) + 1) * Fraction(1, 2 ** 40), (name, m, n, i, j)


def check_contiguous_nn_brute_force(seed=6):
    import oracle
    g = np.random.Generator(np.random.PCG64(seed))
    num_groups, n, k = 2, 128, 128
    m_indices = np.array([1, 1, -1, 0, 0, -1], dtype=np.int32)
    m_total = len(m_indices)
    a = rand_codes(g, (m_total, k))
    b = rand_codes(g, (num_groups, k, n))          # [G][K][N]
    sfa = rand_words(g, m_total, k // 128)
    sfb = np.stack([rand_words(g, 1, k // 128) for _ in range(num_groups)])
    d, written = oracle.m_grouped_fp8_gemm_nn_contiguous(a, sfa, b, sfb, m_indices)
    assert list(written) == [e >= 0 for e in m_indices]
    for i in range(m_total):
        e = m_indices[i]
        if e < 0:
            assert np.all(np.isnan(d[i]))
            continue
        for j in (0, 5, n - 1):
            ex = exact_layout(a, sfa, b[e], sfb[e], None, i, j, False, True)
            assert abs(Fraction(d[i, j]) - ex) <= (abs(ex) + 1) * Fraction(1, 2 ** 40), (i, j)


def check_contiguous_brute_force(seed=1):
    import oracle
    g = np.random.Generator(np.random.PCG64(seed))
    num_groups, n, k = 3, 9, 256
    m_indices = np.array([0, 0, 0, -1, 2, 2, -1, -1, 1, -1], dtype=np.int32)
    m_total = len(m_indices)
    a = rand_codes(g, (m_total, k))
    b = rand_codes(g, (num_groups, n, k))
    sfa = rand_words(g, m_total, k // 128)
    sfb = np.stack([rand_words(g, 1, k // 128) for _ in range(num_groups)])
    d, written = oracle.m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, m_indices)
    assert list(written) == [e >= 0 for e in m_indices]
    for i in range(m_total):
        e = m_indices[i]
        if e < 0:
            assert np.all(np.isnan(d[i]))
            continue
        for j in range(n):
            ex = exact_dense(a, sfa, b[e], sfb[e], None, i, j)
            assert float(ex) == d[i, j] or abs(Fraction(d[i, j]) - ex) <= abs(ex) * Fraction(1, 2 ** 45)


def check_masked_brute_force(seed=2):
    import oracle
    g = np.random.Generator(np.random.PCG64(seed))
    num_groups, m_max, n, k = 3, 6, 5, 256
    masked_m = np.array([0, 6, 2])
    a = rand_codes(g, (num_groups, m_max, k))
    b = rand_codes(g, (num_groups, n, k))
    sfa = np.stack([rand_words(g, m_max, k // 128) for _ in range(num_groups)])
    sfb = np.stack([rand_words(g, 1, k // 128) for _ in range(num_groups)])
    out = oracle.m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, masked_m)
    for e in range(num_groups):
        assert out[e].shape == (masked_m[e], n)
        for i in range(masked_m[e]):
            for j in range(n):
                ex = exact_dense(a[e], sfa[e], b[e], sfb[e], None, i, j)
                assert abs(Fraction(out[e][i, j]) - ex) <= abs(ex) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 900)


def check_k_grouped_brute_force(seed=3):
    import oracle
    g = np.random.Generator(np.random.PCG64(seed))
    m, n = 5, 6
    ks = [256, 0, 128, 384]
    k_total = sum(ks)
    a = rand_codes(g, (k_total, m))
    b = rand_codes(g, (k_total, n))
    sfa = rand_words(g, m, k_total // 128)
    sfb = rand_words(g, n, k_total // 128)
    c = g.standard_normal((len(ks), m, n)).astype(np.float32)
    out = oracle.k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, ks, c)
    assert np.array_equal(out[1], c[1].astype(np.float64))      # empty segment: D = C
    for e in range(len(ks)):
        for i in range(m):
            for j in range(n):
                ex = exact_k_grouped(a, sfa, b, sfb, ks, c, e, i, j)
                assert abs(Fraction(out[e][i, j]) - ex) <= (abs(ex) + 1) * Fraction(1, 2 ** 45)


def check_identity():
    import oracle
    from oracle.formats import pack_ue8m0
    g = np.random.Generator(np.random.PCG64(4))
    a = np.zeros((128, 128), np.uint8)
    np.fill_diagonal(a, 0x38)
    b = rand_codes(g, (200, 128))
    sfa = pack_ue8m0(np.full((128, 1), 127, np.uint8))
    sfb_bytes = np.array([[121], [133]], np.uint8)
    d = oracle.fp8_gemm_nt(a, sfa, b, pack_ue8m0(sfb_bytes))
    want = np.array([[float(fr_e4m3(b[j, i]) * fr_ue8(sfb_bytes[j // 128, 0])) for j in range(200)]
                     for i in range(128)])
    assert np.array_equal(d, want)


def check_one_hot():
    import oracle
    from oracle.formats import pack_ue8m0
    a = np.zeros((4, 256), np.uint8)
    b = np.zeros((3, 256), np.uint8)
    a[2, 200] = 0x4D     # 1.625 * 2^2 = 6.5 ... e=9, m=5
    b[1, 200] = 0xB3     # -(1.375) * 2^-1
    sa = np.full((4, 2), 127, np.uint8)
    sa[2, 1] = 131
    sb = np.full((1, 2), 127, np.uint8)
    sb[0, 1] = 120
    d = oracle.fp8_gemm_nt(a, pack_ue8m0(sa), b, pack_ue8m0(sb))
    want = np.zeros((4, 3))
    want[2, 1] = float(fr_e4m3(0x4D) * fr_e4m3(0xB3) * Fraction(2) ** 4 * Fraction(2) ** -7)
    assert np.array_equal(d, want)
    assert oracle.round_output(d, "bf16")[2, 1] == fr_to_bf16_bits(Fraction(want[2, 1]))


def scale_probe_inputs(m, n, groups):
    """A = B = 1.0 everywhere; scale exponents chosen so that every output is a sum
    of `groups` powers of two whose exponents identify (row, n-block, group)."""
    ea = np.array([[(i * 5 + gg * 7) % 13 - 6 for gg in range(groups)] for i in range(m)])
    eb = np.array([[(j * 3 + gg * 11) % 7 - 3 for gg in range(groups)] for j in range((n + 127) // 128)])
    return ea, eb


def check_scale_probe():
    import oracle
    from oracle.formats import pack_ue8m0
    m, n, groups = 40, 300, 6
    ea, eb = scale_probe_inputs(m, n, groups)
    a = np.full((m, groups * 128), 0x38, np.uint8)
    b = np.full((n, groups * 128), 0x38, np.uint8)
    d = oracle.fp8_gemm_nt(a, pack_ue8m0((ea + 127).astype(np.uint8)), b,
                           pack_ue8m0((eb + 127).astype(np.uint8)))
    for i in range(0, m, 3):
        for j in range(0, n, 17):
            want = sum(Fraction(2) ** (7 + ea[i, gg] + eb[j // 128, gg]) for gg in range(groups))
            assert Fraction(d[i, j]) == want, (i, j)


def check_integer_valued():
    import oracle
    from oracle.formats import pack_ue8m0
    g = np.random.Generator(np.random.PCG64(12))
    vals = {-1: 0xB8, 0: 0x00, 1: 0x38}
    ai = g.integers(-1, 2, (16, 128))
    bi = g.integers(-1, 2, (24, 128))
    a = np.vectorize(vals.get)(ai).astype(np.uint8)
    b = np.vectorize(vals.get)(bi).astype(np.uint8)
    one = pack_ue8m0(np.full((16, 1), 127, np.uint8))
    d = oracle.fp8_gemm_nt(a, one, b, pack_ue8m0(np.full((1, 1), 127, np.uint8)))
    assert np.array_equal(d, (ai @ bi.T).astype(np.float64))


def check_silu_library():
    """SiLU against a library routine (scipy's logistic expit) and its identities."""
    from scipy.special import expit
    from oracle import swiglu as S
    x = np.concatenate([np.linspace(-60, 60, 20001), [0.0, 1e-300, -1e-300, 700.0, -700.0]])
    got = S.silu(x)
    want = x * expit(x)
    assert np.all(np.abs(got - want) <= 4e-16 * np.maximum(np.abs(want), 1e-300))
    assert S.silu(np.array([0.0]))[0] == 0.0
    # silu(x) - silu(-x) = x * (sigma(x) + sigma(-x)) = x
    y = np.linspace(-30, 30, 6001)
    assert np.all(np.abs((S.silu(y) - S.silu(-y)) - y) <= 1e-14 * np.maximum(1.0, np.abs(y)))
    # for x >= 64, exp(-x) is below half an ulp of 1: silu(x) == x exactly in FP64
    z = np.arange(64.0, 200.0)
    assert np.array_equal(S.silu(z), z)


def check_swiglu_brute_force(seed=7):
    """Contiguous gate-up GEMM + SwiGLU + requantisation on a tiny case: the GEMM element
    exactly (rationals), SiLU from scipy's expit, then each code must be the E4M3 value
    nearest to y / scale (half a spacing) and each scale the smallest admissible power of two."""
    from scipy.special import expit
    from oracle import swiglu as S
    g = np.random.Generator(np.random.PCG64(seed))
    num_groups, inter, k = 2, 128, 128
    m_indices = np.array([1, -1, 0, 0], dtype=np.int32)
    a = rand_codes(g, (len(m_indices), k))
    b = rand_codes(g, (num_groups, 2 * inter, k))
    sfa = rand_words(g, len(m_indices), k // 128)
    sfb = np.stack([rand_words(g, 2, k // 128) for _ in range(num_groups)])
    q, sf, written = S.m_grouped_fp8_gemm_nt_contiguous_swiglu(a, sfa, b, sfb, m_indices)
    assert list(written) == [e >= 0 for e in m_indices]
    for r, e in enumerate(m_indices):
        if e < 0:
            continue
        h = np.array([float(exact_dense(a, sfa, b[e], sfb[e], None, r, j)) for j in range(2 * inter)])
        y = (h[:inter] * expit(h[:inter]) * h[inter:]).astype(np.float32).astype(np.float64)
        amax = Fraction(float(np.abs(y).max()))
        scale = fr_ue8(int(sf[r, 0]))
        assert amax <= 448 * scale and (amax == 0 or amax > 224 * scale), (r, float(amax), int(sf[r, 0]))
        for j in range(inter):
            t = Fraction(float(y[j])) / scale
            code = fr_e4m3(int(q[r, j]))
            mag = abs(t)
            ex = max(mag.numerator.bit_length() - mag.denominator.bit_length(), -6) if mag else -6
            if mag and Fraction(2) ** ex > mag:
                ex -= 1
            spacing = Fraction(2) ** (max(ex, -6) - 3)
            assert abs(code - t) <= spacing / 2, (r, j, float(t), float(code))


def check_swiglu_exact_probe():
    """gate >= 64 makes SiLU(gate) == gate, so y = gate * up exactly (small integers): the
    codes and scales then follow from exact arithmetic (torch's E4M3 cast as the library
    rounding of y / scale)."""
    import torch
    from oracle import swiglu as S
    g = np.random.Generator(np.random.PCG64(8))
    gate = g.integers(64, 120, (5, 256)).astype(np.float64)
    up = g.integers(-3, 4, (5, 256)).astype(np.float64)
    q, sf = S.swiglu_quantize(np.concatenate([gate, up], axis=1))
    y = gate * up
    for r in range(5):
        for grp in range(2):
            seg = y[r, grp * 128:(grp + 1) * 128]
            amax = Fraction(int(np.abs(seg).max()))
            e = 0
            while 448 * Fraction(2) ** e < amax:
                e += 1
            while e > -127 and amax and 448 * Fraction(2) ** (e - 1) >= amax:
                e -= 1
            assert int(sf[r, grp]) == (127 if amax == 0 else e + 127), (r, grp)
            ref = torch.from_numpy(seg / 2.0 ** e).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(q[r, grp * 128:(grp + 1) * 128], ref), (r, grp)


def check_mqa_brute_force(seed=9):
    """fp8_mqa_logits against exact rationals, element by element: the kv scale inside
    the dot product, relu per head, the head weights, the [ks, ke) ranges (empty, full,
    clipped past T) and -inf elsewhere."""
    import oracle
    g = np.random.Generator(np.random.PCG64(seed))
    s_len, heads, dim, t_len = 4, 3, 8, 6
    q = rand_codes(g, (s_len, heads, dim))
    kv = rand_codes(g, (t_len, dim))
    sf = (2.0 ** g.integers(-3, 4, t_len)).astype(np.float32)
    w = g.standard_normal((s_len, heads)).astype(np.float32)
    ks = np.array([0, 2, 3, 1]); ke = np.array([6, 5, 3, 9])
    out = oracle.fp8_mqa_logits(q, kv, sf, w, ks, ke, clean_logits=True)
    for i in range(s_len):
        for j in range(t_len):
            if not (ks[i] <= j < min(ke[i], t_len)):
                assert out[i, j] == -np.inf, (i, j)
                continue
            tot = Fraction(0)
            for h in range(heads):
                dot = sum(fr_e4m3(q[i, h, d]) * fr_e4m3(kv[j, d]) * Fraction(float(sf[j])) for d in range(dim))
                tot += max(dot, Fraction(0)) * Fraction(float(w[i, h]))
            assert abs(Fraction(out[i, j]) - tot) <= (abs(tot) + 1) * Fraction(1, 2 ** 44), (i, j)
    kept = oracle.fp8_mqa_logits(q, kv, sf, w, ks, ke, clean_logits=False)
    assert np.isnan(kept[2]).all() and np.isnan(kept[0]).sum() == 0


def check_mqa_closed_form():
    """All-ones q and kv (0x38): every head's dot is D * sf[j] > 0, so
    out[i, j] = D * sf[j] * sum_h w[i, h]; negating q (0xB8) makes every dot negative and
    the logit exactly 0."""
    import oracle
    s_len, heads, dim, t_len = 3, 4, 16, 5
    sf = np.array([1, 2, 0.5, 4, 0.25], np.float32)
    w = np.arange(s_len * heads, dtype=np.float32).reshape(s_len, heads) - 3
    ks, ke = np.zeros(s_len, int), np.full(s_len, t_len)
    ones = oracle.fp8_mqa_logits(np.full((s_len, heads, dim), 0x38, np.uint8), np.full((t_len, dim), 0x38, np.uint8),
                                 sf, w, ks, ke)
    assert np.array_equal(ones, dim * sf[None, :].astype(np.float64) * w.sum(axis=1, dtype=np.float64)[:, None])
    neg = oracle.fp8_mqa_logits(np.full((s_len, heads, dim), 0xB8, np.uint8), np.full((t_len, dim), 0x38, np.uint8),
                                sf, w, ks, ke)
    assert np.array_equal(neg, np.zeros_like(neg))


# ------------------------------------------------------------ FP8 x FP4
GOLDEN_FP4 = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fp4_closed_forms.json")))


def fr_e2m1(code: int) -> Fraction:
    """E2M1 from its bit fields: sign bit 3, exponent bits 1-2 (bias 1), mantissa bit 0."""
    code = int(code)
    s, e, m = code >> 3 & 1, (code >> 1) & 3, code & 1
    mag = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    return -mag if s else mag


def fp4_code(b_row: np.ndarray, kk: int) -> int:
    """Code kk of a packed row: byte kk // 2, low nibble for even kk, high for odd."""
    return (int(b_row[kk // 2]) >> (4 * (kk % 2))) & 0xF


def exact_fp4_dense(a, sfa, b, sfb, c, m, n) -> Fraction:
    """Element (m, n) of C + A @ B.T with A E4M3 (1x128 scales) and B packed E2M1 with one
    scale per 32-block of each row (block j is byte j % 4 of word j // 4)."""
    k = a.shape[1]
    tot = Fraction(0) if c is None else Fraction(float(c[m, n]))
    for kk in range(k):
        tot += (fr_e4m3(a[m, kk]) * fr_ue8(word_byte(sfa, kk // 128, m)) *
                fr_e2m1(fp4_code(b[n], kk)) * fr_ue8(word_byte(sfb, kk // 32, n)))
    return tot


def rand_fp4(g, shape):
    return g.integers(0, 256, shape, dtype=np.uint8)


def check_fp4_format_golden():
    from oracle import fp4
    for row in GOLDEN_FP4["e2m1"]:
        assert fp4.e2m1_to_f64(np.array([int(row["code"], 16)]))[0] == row["value"], row
    for row in GOLDEN_FP4["e2m1_rounding"]:
        assert int(fp4.f64_to_e2m1(np.array([row["x"]]))[0]) == int(row["code"], 16), row


def check_fp4_golden_gemm():
    import oracle
    from oracle.formats import pack_ue8m0
    for case in GOLDEN_FP4["gemm_nt"]:
        m, n, k = case["M"], case["N"], case["K"]
        a = np.empty((m, k), np.uint8)
        a[:, 0::2] = int(case["a_even"], 16)
        a[:, 1::2] = int(case["a_odd"], 16)
        b = np.full((n, k // 2), int(case["b_byte"], 16), np.uint8)
        sfa = pack_ue8m0(np.tile(np.array(case["sa"], np.uint8), (m, 1)))
        sfb = pack_ue8m0(np.tile(np.array(case["sb"], np.uint8), (n, 1)))
        c = None if case["c"] is None else np.full((m, n), case["c"], np.float32)
        d = oracle.fp8_fp4_gemm_nt(a, sfa, b, sfb, c)
        assert np.all(d == case["expect"]), (case["name"], d)


def check_fp4_dense_brute_force(seed=10):
    import oracle
    g = np.random.Generator(np.random.PCG64(seed))
    for (m, n, k, with_c) in [(3, 5, 128, False), (2, 9, 256, True), (4, 3, 384, False)]:
        a, b = rand_codes(g, (m, k)), rand_fp4(g, (n, k // 2))
        sfa, sfb = rand_words(g, m, k // 128), rand_words(g, n, k // 32)
        c = g.standard_normal((m, n)).astype(np.float32) if with_c else None
        d = oracle.fp8_fp4_gemm_nt(a, sfa, b, sfb, c)
        bits = oracle.round_output(d, "bf16")
        for i in range(m):
            for j in range(n):
                ex = exact_fp4_dense(a, sfa, b, sfb, c, i, j)
                mag = sum(abs(fr_e4m3(a[i, kk]) * fr_e2m1(fp4_code(b[j], kk))) for kk in range(k)) * Fraction(2) ** 40
                assert close_fp64(d[i, j], ex, mag, k), (m, n, k, i, j)
                assert bits[i, j] == fr_to_bf16_bits(ex), (i, j)


def check_fp4_grouped_brute_force(seed=11):
    import oracle
    g = np.random.Generator(np.random.PCG64(seed))
    num_groups, n, k = 3, 5, 256
    m_indices = np.array([2, 2, -1, 0, 0, 0, -1, 1], dtype=np.int32)
    m_total = len(m_indices)
    a = rand_codes(g, (m_total, k))
    b = rand_fp4(g, (num_groups, n, k // 2))
    sfa = rand_words(g, m_total, k // 128)
    sfb = np.stack([rand_words(g, n, k // 32) for _ in range(num_groups)])
    d, written = oracle.m_grouped_fp8_fp4_gemm_nt_contiguous(a, sfa, b, sfb, m_indices)
    assert list(written) == [e >= 0 for e in m_indices]
    for i in range(m_total):
        e = m_indices[i]
        if e < 0:
            assert np.all(np.isnan(d[i]))
            continue
        for j in range(n):
            ex = exact_fp4_dense(a, sfa, b[e], sfb[e], None, i, j)
            assert abs(Fraction(d[i, j]) - ex) <= abs(ex) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 900)
    m_max = 4
    masked_m = np.array([3, 0, 4])
    a3 = rand_codes(g, (num_groups, m_max, k))
    sfa3 = np.stack([rand_words(g, m_max, k // 128) for _ in range(num_groups)])
    out = oracle.m_grouped_fp8_fp4_gemm_nt_masked(a3, sfa3, b, sfb, masked_m)
    for e in range(num_groups):
        assert out[e].shape == (masked_m[e], n)
        for i in range(masked_m[e]):
            for j in range(n):
                ex = exact_fp4_dense(a3[e], sfa3[e], b[e], sfb[e], None, i, j)
                assert abs(Fraction(out[e][i, j]) - ex) <= abs(ex) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 900)


def check_fp4_swiglu_brute_force(seed=12):
    """FP4 gate-up GEMM + SwiGLU + requantisation on a tiny case: each GEMM element exactly
    (rationals, nibbles and 1x32 scale bytes read here), SiLU from scipy's expit, then each
    code within half an E4M3 spacing of y / scale and each scale the smallest admissible power
    of two; the masked form on the same weights."""
    from scipy.special import expit
    from oracle import fp4 as FP4
    g = np.random.Generator(np.random.PCG64(seed))
    num_groups, inter, k = 2, 128, 256
    m_indices = np.array([1, -1, 0, 1], dtype=np.int32)
    a = rand_codes(g, (len(m_indices), k))
    b = rand_fp4(g, (num_groups, 2 * inter, k // 2))
    sfa = rand_words(g, len(m_indices), k // 128)
    sfb = np.stack([rand_words(g, 2 * inter, k // 32) for _ in range(num_groups)])
    q, sf, written = FP4.m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(a, sfa, b, sfb, m_indices)
    assert list(written) == [e >= 0 for e in m_indices]

    def check_row(arow_a, arow_sfa, r, e, qrow, sfrow):
        h = np.array([float(exact_fp4_dense(arow_a, arow_sfa, b[e], sfb[e], None, r, j)) for j in range(2 * inter)])
        y = (h[:inter] * expit(h[:inter]) * h[inter:]).astype(np.float32).astype(np.float64)
        amax = Fraction(float(np.abs(y).max()))
        scale = fr_ue8(int(sfrow[0]))
        assert amax <= 448 * scale and (amax == 0 or amax > 224 * scale), (r, float(amax), int(sfrow[0]))
        for j in range(inter):
            t = Fraction(float(y[j])) / scale
            code = fr_e4m3(int(qrow[j]))
            mag = abs(t)
            ex = max(mag.numerator.bit_length() - mag.denominator.bit_length(), -6) if mag else -6
            if mag and Fraction(2) ** ex > mag:
                ex -= 1
            spacing = Fraction(2) ** (max(ex, -6) - 3)
            assert abs(code - t) <= spacing / 2, (r, j, float(t), float(code))

    for r, e in enumerate(m_indices):
        if e >= 0:
            check_row(a, sfa, r, e, q[r], sf[r])
    a3 = a.reshape(2, 2, k)
    sfa3 = np.stack([rand_words(g, 2, k // 128) for _ in range(2)])
    out = FP4.m_grouped_fp8_fp4_gemm_nt_masked_swiglu(a3, sfa3, b, sfb, [2, 1])
    assert out[0][0].shape == (2, inter) and out[1][0].shape == (1, inter)
    for e in range(2):
        for r in range(out[e][0].shape[0]):
            check_row(a3[e], sfa3[e], r, e, out[e][0][r], out[e][1][r])


ALL_CHECKS = [check_golden_gemm, check_dense_brute_force, check_layouts_brute_force,
              check_mqa_brute_force, check_mqa_closed_form,
              check_silu_library, check_swiglu_brute_force, check_swiglu_exact_probe,
              check_contiguous_nn_brute_force, check_contiguous_brute_force,
              check_masked_brute_force, check_k_grouped_brute_force, check_identity,
              check_one_hot, check_scale_probe, check_integer_valued,
              check_fp4_format_golden, check_fp4_golden_gemm, check_fp4_dense_brute_force,
              check_fp4_grouped_brute_force, check_fp4_swiglu_brute_force]
