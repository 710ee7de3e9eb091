"""GPU parity: the CUDA library (through the C ABI) against the oracle, element by
element on the same seeded inputs, plus bit-exact probes and untouched-row checks."""
import numpy as np
import pytest

import cases as C
import oracle_pins as P
from oracle import formats as F

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_fp8_e4m3_gb300 as lib
    return lib


def _status_ok(fg):
    st, detail = fg.get_device_error()
    assert st == 0, (st, hex(detail))


def run_dense(fg, case, alias_c=False):
    from gpu_util import GuardedOut, dev
    out = GuardedOut(case["m"], case["n"], case["out"])
    c_t = None
    if case["c"] is not None:
        if alias_c:
            out.fill_from(case["c"])
            c_t = out.tensor
        else:
            c_t = dev(case["c"])
    fg.fp8_gemm_nt(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]), out.tensor, c=c_t)
    _status_ok(fg)
    out.check_guards()
    return out


# ------------------------------------------------------------------ dense
@pytest.mark.parametrize("m,n,k,with_c,out", [
    (128, 256, 512, False, "bf16"),       # the small dense case
    (200, 272, 384, True, "f32"),         # ragged M and N tails, C
    (1, 16, 128, False, "bf16"),          # minimum sizes
    (64, 512, 1024, True, "f32"),         # decode-like M
    (300, 1000 // 16 * 16, 640, False, "bf16"),
    (513, 384, 2560, True, "f32"),        # K spans several packed scale words
])
def test_dense_parity(fg, m, n, k, with_c, out):
    case = C.dense_case(100 + m + n + k, m, n, k, with_c, out)
    got = run_dense(fg, case)
    C.compare(got.values(), C.dense_ref(case), f"dense {m}x{n}x{k}")


@pytest.mark.parametrize("bn", ["64", "128", "192", "224", "256"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_dense_every_tile_width(fg, bn, out, monkeypatch):
    monkeypatch.setenv("FG_FORCE_BN", bn)
    case = C.dense_case(7, 300, 784, 1024, out == "f32", out)   # ragged M and N, several tiles each
    got = run_dense(fg, case)
    C.compare(got.values(), C.dense_ref(case), f"BN={bn} {out}")


@pytest.mark.parametrize("bn", ["64", "128", "192", "224", "256"])
def test_grouped_every_tile_width(fg, bn, monkeypatch):
    monkeypatch.setenv("FG_FORCE_BN", bn)
    case = C.contiguous_case(9, num_tokens=512, num_routed=16, topk=3, num_groups=5, n=448, k=256)
    d = run_contiguous(fg, case)
    ref, written = C.contiguous_ref(case)
    assert np.array_equal(~d.is_sentinel(), written)
    C.compare(d.values()[written], ref[written], f"contiguous BN={bn}")
    mc = C.masked_case(10, num_groups=3, m_max=160, n=448, k=256, masked_m=[0, 97, 160])
    _check_masked(mc, run_masked(fg, mc))


@pytest.mark.parametrize("bn", ["128", "256"])
def test_k_grouped_every_tile_width(fg, bn, monkeypatch):
    monkeypatch.setenv("FG_FORCE_BN", bn)
    case = C.k_grouped_case(11, num_groups=3, m=256, n=384, ks=[256, 128, 0])
    d = run_k_grouped(fg, case)
    ref = C.k_grouped_ref(case)
    vals = d.values().reshape(case["g"], case["m"], case["n"])
    for e in range(case["g"]):
        C.compare(vals[e], ref[e], f"k-grouped BN={bn} group {e}")


def test_dense_d_aliases_c(fg):
    case = C.dense_case(8, 256, 256, 256, True, "f32")
    got = run_dense(fg, case, alias_c=True)
    C.compare(got.values(), C.dense_ref(case), "aliased C")


@pytest.mark.parametrize("bn,split", [("224", "1"), ("256", "1"), ("128", "1"), ("128", "2")])
def test_dense_in_place_every_form(fg, bn, split, monkeypatch):
    """D aliasing C (in-place accumulation) in the one-CTA kernels, where the product is
    added onto D by TMA reduce-adds (tile widths with and without C slots), and in a
    split-K cluster, where each thread reads C and writes D."""
    monkeypatch.setenv("FG_FORCE_BN", bn)
    monkeypatch.setenv("FG_FORCE_SPLIT", split)
    case = C.dense_case(811, 300, 528, 640, True, "f32")
    got = run_dense(fg, case, alias_c=True)
    C.compare(got.values(), C.dense_ref(case), f"in place BN={bn} split={split}")


def test_scale_identification_probe_bit_exact(fg):
    """A = B = 1.0; every (row, group) and (n-block, group) scale is a distinct power of
    two, so each FP32 output names exactly which scales were applied."""
    from gpu_util import GuardedOut, dev
    m, n, groups = 256, 512, 8
    ea, eb = P.scale_probe_inputs(m, n, groups)
    a = np.full((m, groups * 128), 0x38, np.uint8)
    b = np.full((n, groups * 128), 0x38, np.uint8)
    sfa = F.pack_ue8m0((ea + 127).astype(np.uint8))
    sfb = F.pack_ue8m0((eb + 127).astype(np.uint8))
    out = GuardedOut(m, n, "f32")
    fg.fp8_gemm_nt(dev(a), dev(sfa), dev(b), dev(sfb), out.tensor)
    _status_ok(fg)
    want = np.zeros((m, n))
    for gg in range(groups):
        want += 2.0 ** (7 + ea[:, gg][:, None] + eb[np.arange(n) // 128, gg][None, :])
    got = out.values()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}: got {got[tuple(bad[0])]} want {want[tuple(bad[0])]}"


def test_integer_valued_bit_exact(fg):
    from gpu_util import GuardedOut, dev
    g = np.random.Generator(np.random.PCG64(12))
    codes = np.array([0xB8, 0x00, 0x38], np.uint8)          # -1, 0, 1
    ai = g.integers(-1, 2, (160, 128))
    bi = g.integers(-1, 2, (96, 128))
    a, b = codes[ai + 1], codes[bi + 1]
    sfa = F.pack_ue8m0(np.full((160, 1), 127, np.uint8))
    sfb = F.pack_ue8m0(np.full((1, 1), 127, np.uint8))
    out = GuardedOut(160, 96, "bf16")
    fg.fp8_gemm_nt(dev(a), dev(sfa), dev(b), dev(sfb), out.tensor)
    _status_ok(fg)
    assert np.array_equal(out.values(), (ai @ bi.T).astype(np.float64))


def test_identity_bit_exact(fg):
    from gpu_util import GuardedOut, dev
    g = np.random.Generator(np.random.PCG64(4))
    a = np.zeros((128, 128), np.uint8)
    np.fill_diagonal(a, 0x38)
    b = P.rand_codes(g, (256, 128))
    sfb_bytes = np.array([[121], [133]], np.uint8)
    out = GuardedOut(128, 256, "bf16")
    fg.fp8_gemm_nt(dev(a), dev(F.pack_ue8m0(np.full((128, 1), 127, np.uint8))), dev(b),
                   dev(F.pack_ue8m0(sfb_bytes)), out.tensor)
    _status_ok(fg)
    want = (F.e4m3_to_f64(b) * F.ue8m0_to_f64(sfb_bytes[np.arange(256) // 128])).T
    assert np.array_equal(out.values(), want)


# ------------------------------------------------------------- contiguous
def run_contiguous(fg, case, out="bf16"):
    from gpu_util import GuardedOut, dev
    d = GuardedOut(case["m_total"], case["n"], out)
    fg.m_grouped_fp8_gemm_nt_contiguous(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                        dev(case["m_indices"]), d.tensor)
    _status_ok(fg)
    d.check_guards()
    return d


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_contiguous_parity(fg, out):
    case = C.contiguous_case(2, num_tokens=512, num_routed=16, topk=3, num_groups=5, n=256, k=384)
    d = run_contiguous(fg, case, out)
    ref, written = C.contiguous_ref(case)
    assert np.array_equal(~d.is_sentinel(), written), "written row set differs"
    C.compare(d.values()[written], ref[written], "contiguous")


def test_contiguous_empty_groups_and_all_padding_block(fg):
    # group 1 receives no tokens; the last block is all padding
    g = np.random.Generator(np.random.PCG64(31))
    m_indices = np.array([0] * 130 + [-1] * 126 + [2] * 128 + [-1] * 128, np.int32)
    k, n, groups = 256, 128, 3
    a = P.rand_codes(g, (len(m_indices), k))
    b = P.rand_codes(g, (groups, n, k))
    sfa = P.rand_words(g, len(m_indices), k // 128)
    sfb = np.stack([P.rand_words(g, 1, k // 128) for _ in range(groups)])
    case = {"m_total": len(m_indices), "n": n, "k": k, "g": groups, "a": a, "sfa": sfa, "b": b,
            "sfb": sfb, "m_indices": m_indices}
    d = run_contiguous(fg, case)
    ref, written = C.contiguous_ref(case)
    assert np.array_equal(~d.is_sentinel(), written)
    C.compare(d.values()[written], ref[written], "contiguous edge")


def test_contiguous_contract_violation_reported(fg):
    from gpu_util import GuardedOut, dev
    g = np.random.Generator(np.random.PCG64(32))
    m_indices = np.array([0] * 128 + [5] * 128, np.int32)   # group 5 >= G
    k, n = 128, 64
    a = P.rand_codes(g, (256, k))
    b = P.rand_codes(g, (2, n, k))
    d = GuardedOut(256, n, "bf16")
    fg.m_grouped_fp8_gemm_nt_contiguous(dev(a), dev(P.rand_words(g, 256, 1)), dev(b),
                                        dev(np.stack([P.rand_words(g, 1, 1)] * 2)), dev(m_indices), d.tensor)
    st, detail = fg.get_device_error()
    assert st == fg.FG_ERR_DEVICE_CONTRACT and detail == 0x101
    assert np.all(d.is_sentinel()[128:]) and not np.any(d.is_sentinel()[:128])


def test_contiguous_padding_first_block_naming_a_group_reported(fg):
    """A block whose first row is padding (-1) is skipped; if a later row of it names a
    group the layout is malformed (segments must start on 128-row boundaries): the call
    reports it (0x102) and leaves the whole block untouched."""
    from gpu_util import GuardedOut, dev
    g = np.random.Generator(np.random.PCG64(33))
    m_indices = np.array([0] * 128 + [-1] * 5 + [1] * 123 + [1] * 128, np.int32)
    k, n = 256, 128
    a = P.rand_codes(g, (len(m_indices), k))
    b = P.rand_codes(g, (2, n, k))
    sfa = P.rand_words(g, len(m_indices), k // 128)
    sfb = np.stack([P.rand_words(g, 1, k // 128) for _ in range(2)])
    d = GuardedOut(len(m_indices), n, "bf16")
    fg.m_grouped_fp8_gemm_nt_contiguous(dev(a), dev(sfa), dev(b), dev(sfb), dev(m_indices), d.tensor)
    st, detail = fg.get_device_error()
    assert st == fg.FG_ERR_DEVICE_CONTRACT and detail == 0x102, (st, hex(detail))
    d.check_guards()
    sent = d.is_sentinel()
    assert np.all(sent[128:256]) and not np.any(sent[:128]) and not np.any(sent[256:])
    case = {"m_total": len(m_indices), "n": n, "k": k, "g": 2, "a": a, "sfa": sfa, "b": b, "sfb": sfb,
            "m_indices": m_indices}
    ref, _ = C.contiguous_ref(case)
    vals = d.values()
    C.compare(vals[:128], ref[:128], "block 0")
    C.compare(vals[256:], ref[256:], "block 2")


# ----------------------------------------------------------------- masked
def run_masked(fg, case, out="bf16"):
    from gpu_util import GuardedOut, dev
    d = GuardedOut(case["g"] * case["m_max"], case["n"], out)
    fg.m_grouped_fp8_gemm_nt_masked(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                    dev(case["masked_m"]), d.tensor.view(case["g"], case["m_max"], case["n"]))
    _status_ok(fg)
    d.check_guards()
    return d


def _check_masked(case, d):
    ref = C.masked_ref(case)
    vals = d.values().reshape(case["g"], case["m_max"], case["n"])
    sent = d.is_sentinel().reshape(case["g"], case["m_max"])
    for e in range(case["g"]):
        mm = int(case["masked_m"][e])
        assert not sent[e, :mm].any() and sent[e, mm:].all(), f"group {e}: rows beyond mask written"
        if mm:
            C.compare(vals[e, :mm], ref[e], f"masked group {e}")


@pytest.mark.parametrize("masks", [[0, 1, 192, 100], [128, 129, 64, 0]])
def test_masked_parity(fg, masks):
    case = C.masked_case(3, num_groups=4, m_max=192, n=256, k=384, masked_m=masks)
    _check_masked(case, run_masked(fg, case))


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_masked_m_max_not_multiple_of_32(fg, out):
    """M_max = 200: the second 128-row block of a group reaches into the next group's rows
    (or past the end of A for the last group); only rows below the mask are written, and
    masks cover 0, 1, 31, 32, 127, 128, 129, 199 and 200 rows."""
    masks = [0, 1, 31, 32, 127, 128, 129, 199, 200]
    case = C.masked_case(8, num_groups=len(masks), m_max=200, n=272, k=384, masked_m=masks)
    _check_masked(case, run_masked(fg, case, out))


def test_masked_random_masks(fg):
    case = C.masked_case(4, num_groups=6, m_max=256, n=384, k=256)
    _check_masked(case, run_masked(fg, case))


# -------------------------------------------------------------- K-grouped
def run_k_grouped(fg, case, alias_c=False):
    from gpu_util import GuardedOut, dev
    g, m, n = case["g"], case["m"], case["n"]
    d = GuardedOut(g * m, n, "f32")
    c_t = None
    if case["c"] is not None:
        if alias_c:
            d.fill_from(case["c"].reshape(g * m, n))
            c_t = d.tensor.view(g, m, n)
        else:
            c_t = dev(case["c"])
    fg.k_grouped_fp8_gemm_tn_contiguous(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                        dev(case["ks"]), d.tensor.view(g, m, n), c=c_t)
    _status_ok(fg)
    d.check_guards()
    return d


@pytest.mark.parametrize("bn", ["128", "256"])
def test_k_grouped_in_place_tile_widths(fg, bn, monkeypatch):
    """K-grouped accumulation into C itself (TMA reduce-adds) at both tile widths, with an
    empty segment (its D must stay exactly C)."""
    monkeypatch.setenv("FG_FORCE_BN", bn)
    case = C.k_grouped_case(812, num_groups=3, m=256, n=384, ks=[384, 0, 256])
    d = run_k_grouped(fg, case, alias_c=True)
    ref = C.k_grouped_ref(case)
    vals = d.values().reshape(case["g"], case["m"], case["n"])
    for e in range(case["g"]):
        C.compare(vals[e], ref[e], f"k-grouped in place BN={bn} group {e}")
    assert np.array_equal(vals[1].astype(np.float32), case["c"][1])


@pytest.mark.parametrize("alias_c", [False, True])
def test_k_grouped_parity(fg, alias_c):
    case = C.k_grouped_case(5, num_groups=4, m=256, n=384, ks=[200, 0, 128, 300])
    d = run_k_grouped(fg, case, alias_c)
    ref = C.k_grouped_ref(case)
    vals = d.values().reshape(case["g"], case["m"], case["n"])
    for e in range(case["g"]):
        C.compare(vals[e], ref[e], f"k-grouped group {e}")
    # the empty segment copies C exactly
    assert np.array_equal(vals[1], case["c"][1].astype(np.float64))


def test_k_grouped_without_c_and_ragged_m(fg):
    case = C.k_grouped_case(6, with_c=False, num_groups=3, m=208, n=144, ks=[128, 384, 5])
    d = run_k_grouped(fg, case)
    ref = C.k_grouped_ref(case)
    vals = d.values().reshape(case["g"], case["m"], case["n"])
    for e in range(case["g"]):
        C.compare(vals[e], ref[e], f"k-grouped group {e}")


def test_k_grouped_bad_segments_reported(fg):
    from gpu_util import GuardedOut, dev
    case = C.k_grouped_case(7, num_groups=2, m=128, n=128, ks=[128, 128])
    d = GuardedOut(2 * 128, 128, "f32")
    bad_ks = np.array([128, 64], np.int32)            # not a multiple of 128, wrong sum
    fg.k_grouped_fp8_gemm_tn_contiguous(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                        dev(bad_ks), d.tensor.view(2, 128, 128), c=dev(case["c"]))
    st, detail = fg.get_device_error()
    assert st == fg.FG_ERR_DEVICE_CONTRACT and detail == 0x104
    assert np.all(d.is_sentinel())


# ------------------------------------------------------------ split-K clusters
def _launched_split(capfd):
    err = capfd.readouterr().err
    lines = [ln for ln in err.splitlines() if ln.startswith("[fg] fp8_gemm_nt")]
    assert lines, err
    return int(lines[-1].split("split=")[1].split()[0])


@pytest.mark.parametrize("split", ["2", "4", "8"])
@pytest.mark.parametrize("bn,out,with_c", [
    ("64", "f32", True), ("128", "bf16", False), ("192", "f32", True), ("224", "bf16", False),
    ("256", "f32", True),
])
@pytest.mark.parametrize("m,n,k", [
    (100, 800, 1280),     # one ragged row block, N tail, 10 K-groups (uneven shares)
    (40, 480, 640),       # <= 64 rows (64-row A box); 5 K-groups: with 8 CTAs some run none
])
def test_dense_split_k(fg, split, bn, out, with_c, m, n, k, monkeypatch, capfd):
    """Split-K clusters: the CTAs of a cluster share one tile along K and sum their
    partial tiles through distributed shared memory."""
    monkeypatch.setenv("FG_FORCE_SPLIT", split)
    monkeypatch.setenv("FG_FORCE_BN", bn)
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    case = C.dense_case(71 + m + int(bn) + int(split), m, n, k, with_c, out)
    got = run_dense(fg, case)
    assert _launched_split(capfd) == int(split)
    C.compare(got.values(), C.dense_ref(case), f"split-K {split} BN={bn} {m}x{n}x{k}")


def test_dense_split_k_aliased_c(fg, monkeypatch, capfd):
    monkeypatch.setenv("FG_FORCE_SPLIT", "4")
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    case = C.dense_case(83, 64, 1024, 2048, True, "f32")
    got = run_dense(fg, case, alias_c=True)
    assert _launched_split(capfd) == 4
    C.compare(got.values(), C.dense_ref(case), "split-K aliased C")


@pytest.mark.parametrize("split", ["2", "4"])
def test_scale_probe_split_k(fg, split, monkeypatch, capfd):
    """The scale-identification probe under a K split: partial sums of distinct powers
    of two stay exact, so the result is still bit-exact."""
    from gpu_util import GuardedOut, dev
    monkeypatch.setenv("FG_FORCE_SPLIT", split)
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    m, n, groups = 120, 512, 8
    ea, eb = P.scale_probe_inputs(m, n, groups)
    a = np.full((m, groups * 128), 0x38, np.uint8)
    b = np.full((n, groups * 128), 0x38, np.uint8)
    out = GuardedOut(m, n, "f32")
    fg.fp8_gemm_nt(dev(a), dev(F.pack_ue8m0((ea + 127).astype(np.uint8))), dev(b),
                   dev(F.pack_ue8m0((eb + 127).astype(np.uint8))), out.tensor)
    _status_ok(fg)
    out.check_guards()
    assert _launched_split(capfd) == int(split)
    want = np.zeros((m, n))
    for gg in range(groups):
        want += 2.0 ** (7 + ea[:, gg][:, None] + eb[np.arange(n) // 128, gg][None, :])
    assert np.array_equal(out.values(), want)


# ------------------------------------------- programmatic dependent launch order
def _gemm(fg, case, d, c=None):
    from gpu_util import dev
    fg.fp8_gemm_nt(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]), d, c=c)


def _chain(fg, pdl):
    """Back-to-back GEMMs with no host synchronisation between them.
    Read after write: a slow GEMM (K=4096) writes X, then a fast one (K=128) reads X as C.
    Write after read: a slow GEMM reads X2 as C, then a fast one overwrites X2.
    X and X2 start as NaN sentinels, so any premature read or write shows."""
    from gpu_util import GuardedOut, dev
    fg.set_pdl(pdl)
    m, n = 512, 1024
    slow = C.dense_case(91, m, n, 4096, False, "f32")
    fast = C.dense_case(92, m, n, 128, True, "f32")
    x, y = GuardedOut(m, n, "f32"), GuardedOut(m, n, "f32")
    x2, y2 = GuardedOut(m, n, "f32"), GuardedOut(m, n, "f32")
    x2.fill_from(fast["c"])
    ops = [dev(t) for t in (slow["a"], slow["sfa"], slow["b"], slow["sfb"], fast["a"], fast["sfa"],
                            fast["b"], fast["sfb"])]
    torch.cuda.synchronize()
    fg.fp8_gemm_nt(ops[0], ops[1], ops[2], ops[3], x.tensor)                  # X = slow
    fg.fp8_gemm_nt(ops[4], ops[5], ops[6], ops[7], y.tensor, c=x.tensor)      # Y = X + fast
    fg.fp8_gemm_nt(ops[0], ops[1], ops[2], ops[3], y2.tensor, c=x2.tensor)    # Y2 = X2 + slow
    fg.fp8_gemm_nt(ops[4], ops[5], ops[6], ops[7], x2.tensor)                 # X2 = fast (no C)
    _status_ok(fg)
    for g in (x, y, x2, y2):
        g.check_guards()
    return slow, fast, x, y, x2, y2


def test_pdl_dependent_launch_order(fg):
    try:
        slow, fast, x, y, x2, y2 = _chain(fg, True)
        rows = np.array([0, 1, 127, 128, 300, 511])
        slow_ref = C.dense_ref(slow, rows=rows)
        fast_nc = dict(fast, c=None)
        fast_ref = C.dense_ref(fast_nc, rows=rows)
        C.compare(x.values()[rows], slow_ref, "X = slow")
        C.compare(y.values()[rows], slow_ref + fast_ref, "Y = X + fast (read after write)")
        C.compare(y2.values()[rows], fast["c"][rows] + slow_ref, "Y2 = X2 + slow (write after read)")
        C.compare(x2.values()[rows], fast_ref, "X2 = fast")
        # results never depend on the launch mode
        bits_on = [g.inner_bits().copy() for g in (x, y, x2, y2)]
        _, _, *outs_off = _chain(fg, False)
        for a, g in zip(bits_on, outs_off):
            assert np.array_equal(a, g.inner_bits())
    finally:
        fg.set_pdl(True)


# ------------------------------------------------------- NN / TN / TT layouts
def run_layout(fg, case, alias_c=False):
    from gpu_util import GuardedOut, dev
    out = GuardedOut(case["m"], case["n"], case["out"])
    c_t = None
    if case["c"] is not None:
        if alias_c:
            out.fill_from(case["c"])
            c_t = out.tensor
        else:
            c_t = dev(case["c"])
    fn = {"nn": fg.fp8_gemm_nn, "tn": fg.fp8_gemm_tn, "tt": fg.fp8_gemm_tt}[case["layout"]]
    fn(dev(case["a_stored"]), dev(case["sfa"]), dev(case["b_stored"]), dev(case["sfb"]), out.tensor, c=c_t)
    _status_ok(fg)
    out.check_guards()
    return out


@pytest.mark.parametrize("layout,bn", [(lay, bn) for lay in ("nn", "tn", "tt") for bn in ("128", "256")]
                         + [("tt", "224")])
@pytest.mark.parametrize("m,n,k,with_c,out", [
    (128, 256, 512, False, "bf16"),
    (208, 272, 384, True, "f32"),         # ragged M and N tails, C
    (64, 512, 1024, True, "f32"),         # one row block of 64 rows
    (512, 400, 1280, False, "bf16"),      # several row blocks, N tail inside a 256 tile
])
def test_dense_layouts(fg, layout, bn, m, n, k, with_c, out, monkeypatch):
    """fp8_gemm_{nn,tn,tt}: the same product with A stored [K, M] ("t") and/or B stored
    [K, N] ("n"); MN-major operands go through 128-wide swizzle atoms in shared memory."""
    monkeypatch.setenv("FG_FORCE_BN", bn)
    case = C.layout_case(300 + m + n + k, layout, m, n, k, with_c, out)
    C.compare(run_layout(fg, case).values(), C.layout_ref(case), f"{layout} BN={bn} {m}x{n}x{k}")


def test_dense_layout_aliased_c(fg):
    case = C.layout_case(41, "tn", 256, 384, 640, True, "f32")
    C.compare(run_layout(fg, case, alias_c=True).values(), C.layout_ref(case), "tn aliased C")


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
def test_layouts_match_nt_bit_for_bit(fg, layout, monkeypatch):
    """Only the operand storage differs from NT (no K split): same values, same
    accumulation order, so the FP32 outputs agree bit for bit."""
    monkeypatch.setenv("FG_FORCE_SPLIT", "1")
    case = C.layout_case(43, layout, 256, 512, 1024, True, "f32")
    got = run_layout(fg, case).inner_bits()
    nt = run_dense(fg, case).inner_bits()
    assert np.array_equal(got, nt)


@pytest.mark.parametrize("bn", ["128", "256"])
def test_contiguous_nn_parity(fg, bn, monkeypatch):
    """m_grouped_fp8_gemm_nn_contiguous: expert weights stored [G, K, N]."""
    from gpu_util import GuardedOut, dev
    monkeypatch.setenv("FG_FORCE_BN", bn)
    case = C.contiguous_case(7, num_tokens=512, num_routed=16, topk=3, num_groups=5, n=384, k=384)
    b_nn = np.ascontiguousarray(np.transpose(case["b"], (0, 2, 1)))
    d = GuardedOut(case["m_total"], case["n"], "bf16")
    fg.m_grouped_fp8_gemm_nn_contiguous(dev(case["a"]), dev(case["sfa"]), dev(b_nn), dev(case["sfb"]),
                                        dev(case["m_indices"]), d.tensor)
    _status_ok(fg)
    d.check_guards()
    ref, written = C.oracle.m_grouped_fp8_gemm_nn_contiguous(case["a"], case["sfa"], b_nn, case["sfb"],
                                                             case["m_indices"])
    assert np.array_equal(~d.is_sentinel(), written), "written row set differs"
    C.compare(d.values()[written], ref[written], f"contiguous nn BN={bn}")
