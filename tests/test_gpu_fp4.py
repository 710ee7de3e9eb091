"""GPU parity of the FP8 x FP4 GEMMs (E4M3 activations with 1x128 scales, packed E2M1 weights
with one UE8M0 scale per 32 K elements of a row) against the oracle, through the C ABI:
bit-exact probes of the nibble order and of the scale-byte selection, element-wise parity
across shapes, tile widths, split-K clusters, in-place C and the M-grouped layouts."""
import numpy as np
import pytest

import cases as C
from oracle import formats as F
from oracle import fp4 as FP4

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


def run_fp4_dense(fg, case, alias_c=False):
    from gpu_util import GuardedOut, dev
    out = GuardedOut(case["m"], case["n"], case["out"])
    c_t = None
    if case["c"] is not None:
        if alias_c:
            out.fill_from(case["c"])
            c_t = out.tensor
        else:
            c_t = dev(case["c"])
    fg.fp8_fp4_gemm_nt(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]), out.tensor, c=c_t)
    _status_ok(fg)
    out.check_guards()
    return out


def _launched(capfd, prefix):
    err = capfd.readouterr().err
    lines = [ln for ln in err.splitlines() if ln.startswith("[fg] " + prefix)]
    assert lines, err
    return dict(kv.split("=") for kv in lines[-1].split()[2:])


# ------------------------------------------------------------------ probes
def test_fp4_nibble_order_probe(fg):
    """A is 1 at even k and 2 at odd k; every byte of B is 0xA7 (low nibble 6, high nibble
    -1): each pair adds 6 - 2 = 4, so D = 2K exactly (the swapped order would give 5.5 K)."""
    from gpu_util import GuardedOut, dev
    m, n, k = 128, 64, 256
    a = np.empty((m, k), np.uint8)
    a[:, 0::2], a[:, 1::2] = 0x38, 0x40
    b = np.full((n, k // 2), 0xA7, np.uint8)
    sfa = F.pack_ue8m0(np.full((m, k // 128), 127, np.uint8))
    sfb = FP4.pack_mx_scales(np.full((n, k // 32), 127, np.uint8))
    out = GuardedOut(m, n, "f32")
    fg.fp8_fp4_gemm_nt(dev(a), dev(sfa), dev(b), dev(sfb), out.tensor)
    _status_ok(fg)
    assert np.array_equal(out.values(), np.full((m, n), 2.0 * k))


@pytest.mark.parametrize("bn", ["128", "224"])
def test_fp4_scale_selection_probe(fg, bn, monkeypatch):
    """Every code 1.0; A's scale varies with row and K-group, B's with row and 32-wide block,
    so every output is a distinct exact sum of powers of two: a wrong byte, word or row of
    either scale array changes it."""
    from gpu_util import GuardedOut, dev
    monkeypatch.setenv("FG_FORCE_BN", bn)
    m, n, k = 200, 288, 768
    sa = (126 + (np.arange(m)[:, None] + np.arange(k // 128)[None, :]) % 3).astype(np.uint8)
    sb = (124 + (np.arange(n)[:, None] + 3 * np.arange(k // 32)[None, :]) % 7).astype(np.uint8)
    a = np.full((m, k), 0x38, np.uint8)
    b = np.full((n, k // 2), 0x22, np.uint8)
    out = GuardedOut(m, n, "f32")
    fg.fp8_fp4_gemm_nt(dev(a), dev(F.pack_ue8m0(sa)), dev(b), dev(FP4.pack_mx_scales(sb)), out.tensor)
    _status_ok(fg)
    want = 32.0 * (np.repeat(np.exp2(sa - 127.0), 4, axis=1) @ np.exp2(sb - 127.0).T)
    assert np.array_equal(out.values(), want)


# ------------------------------------------------------------------- dense
@pytest.mark.parametrize("m,n,k,with_c,out", [
    (128, 256, 512, False, "bf16"),
    (200, 272, 384, True, "f32"),         # ragged M and N tails, C
    (1, 16, 128, False, "bf16"),          # minimum sizes
    (64, 512, 1024, True, "f32"),         # decode-like M
    (513, 384, 2560, True, "f32"),        # K spans several scale word rows
])
def test_fp4_dense_parity(fg, m, n, k, with_c, out):
    case = C.fp4_dense_case(400 + m + n + k, m, n, k, with_c, out)
    got = run_fp4_dense(fg, case)
    C.compare(got.values(), C.fp4_dense_ref(case), f"fp4 dense {m}x{n}x{k}")


@pytest.mark.parametrize("bn", ["128", "224"])
@pytest.mark.parametrize("out,with_c", [("f32", True), ("bf16", False), ("f32", False)])
def test_fp4_dense_every_tile_width(fg, bn, out, with_c, monkeypatch, capfd):
    monkeypatch.setenv("FG_FORCE_BN", bn)
    monkeypatch.setenv("FG_FORCE_SPLIT", "1")
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    case = C.fp4_dense_case(17, 300, 784, 1024, with_c, out)
    got = run_fp4_dense(fg, case)
    assert _launched(capfd, "fp8_fp4_gemm_nt")["BN"] == bn
    C.compare(got.values(), C.fp4_dense_ref(case), f"fp4 BN={bn} {out}")


@pytest.mark.parametrize("split", ["1", "2"])
def test_fp4_dense_d_aliases_c(fg, split, monkeypatch):
    monkeypatch.setenv("FG_FORCE_SPLIT", split)
    case = C.fp4_dense_case(18, 96, 512, 1024, True, "f32")
    got = run_fp4_dense(fg, case, alias_c=True)
    C.compare(got.values(), C.fp4_dense_ref(case), f"fp4 in place split={split}")


@pytest.mark.parametrize("split", ["2", "4", "8"])
@pytest.mark.parametrize("m,n,k,with_c,out", [
    (100, 800, 1280, True, "f32"),        # ragged rows and N, 10 K-groups (uneven shares)
    (40, 480, 640, False, "bf16"),        # <= 64 rows; 5 K-groups: with 8 CTAs some run none
])
def test_fp4_dense_split_k(fg, split, m, n, k, with_c, out, monkeypatch, capfd):
    monkeypatch.setenv("FG_FORCE_SPLIT", split)
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    case = C.fp4_dense_case(19 + int(split) + m, m, n, k, with_c, out)
    got = run_fp4_dense(fg, case)
    cfg = _launched(capfd, "fp8_fp4_gemm_nt")
    assert cfg["split"] == split and cfg["BN"] == "128", cfg
    C.compare(got.values(), C.fp4_dense_ref(case), f"fp4 split-K {split} {m}x{n}x{k}")


def test_fp4_decode_shape(fg):
    """The decode shape 64 x 7168 x 4096 with FP32 C, as the cost model tiles it; rows
    compared element by element."""
    case = C.fp4_dense_case(20, 64, 7168, 4096, True, "f32")
    got = run_fp4_dense(fg, case)
    C.compare(got.values(), C.fp4_dense_ref(case), "fp4 decode")


# --------------------------------------------------------------- M-grouped
def run_fp4_contiguous(fg, case, out="bf16"):
    from gpu_util import GuardedOut, dev
    d = GuardedOut(case["m_total"], case["n"], out)
    fg.m_grouped_fp8_fp4_gemm_nt_contiguous(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                            dev(case["m_indices"]), d.tensor)
    _status_ok(fg)
    d.check_guards()
    return d


def run_fp4_masked(fg, case, out="bf16"):
    from gpu_util import GuardedOut, dev
    d = GuardedOut(case["g"] * case["m_max"], case["n"], out)
    fg.m_grouped_fp8_fp4_gemm_nt_masked(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                        dev(case["masked_m"]), d.tensor.view(case["g"], case["m_max"], case["n"]))
    _status_ok(fg)
    d.check_guards()
    return d


@pytest.mark.parametrize("bn", ["128", "224"])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_fp4_contiguous_parity(fg, bn, out, monkeypatch):
    monkeypatch.setenv("FG_FORCE_BN", bn)
    case = C.fp4_contiguous_case(21, num_tokens=512, num_routed=16, topk=3, num_groups=5, n=448, k=384)
    d = run_fp4_contiguous(fg, case, out)
    ref, written = C.fp4_contiguous_ref(case)
    assert np.array_equal(~d.is_sentinel(), written), "written row set differs"
    C.compare(d.values()[written], ref[written], f"fp4 contiguous BN={bn}")


@pytest.mark.parametrize("bn", ["128", "224"])
def test_fp4_masked_parity(fg, bn, monkeypatch):
    monkeypatch.setenv("FG_FORCE_BN", bn)
    masks = [0, 1, 31, 128, 129, 200]
    case = C.fp4_masked_case(22, num_groups=len(masks), m_max=200, n=448, k=512, masked_m=masks)
    d = run_fp4_masked(fg, case)
    ref = C.fp4_masked_ref(case)
    vals = d.values().reshape(case["g"], case["m_max"], case["n"])
    sent = d.is_sentinel().reshape(case["g"], case["m_max"])
    for e, mm in enumerate(masks):
        assert not sent[e, :mm].any() and sent[e, mm:].all(), f"group {e}: rows beyond mask written"
        if mm:
            C.compare(vals[e, :mm], ref[e], f"fp4 masked BN={bn} group {e}")


# ----------------------------------------------- FP4 gate-up GEMM + SwiGLU
SENT_Q = 0xAB
SENT_W = -0x21436588


def _y_ref(h):
    from oracle import swiglu as S
    return S.swiglu(h).astype(np.float32).astype(np.float64)


def test_fp4_contiguous_swiglu_parity(fg):
    """The Mega MoE's linear 1 in FP8 x FP4 with the fused SwiGLU + requantisation (same
    comparison rule as the E4M3-weight form: one E4M3 spacing, >= 99 % identical codes)."""
    from gpu_util import dev
    from oracle import swiglu as S
    inter = 256
    case = C.fp4_contiguous_case(31, num_tokens=512, num_routed=16, topk=3, num_groups=5, n=2 * inter, k=384)
    m_total = case["m_total"]
    q = torch.full((m_total, inter), SENT_Q, dtype=torch.uint8, device="cuda")
    sfq = torch.full(((inter + 511) // 512, (m_total + 3) // 4 * 4), SENT_W, dtype=torch.int32, device="cuda")
    fg.m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(dev(case["a"]), dev(case["sfa"]), dev(case["b"]),
                                                   dev(case["sfb"]), dev(case["m_indices"]), q, sfq)
    _status_ok(fg)
    qh, sfh = q.cpu().numpy(), sfq.cpu().numpy()
    written = case["m_indices"] >= 0
    assert np.all(qh[~written] == SENT_Q), "padding rows of q written"
    sf_bytes = F.unpack_ue8m0(sfh, m_total, inter // 128)
    sent_bytes = F.unpack_ue8m0(np.full_like(sfh, SENT_W), m_total, inter // 128)
    assert np.array_equal(sf_bytes[~written], sent_bytes[~written]), "padding rows of sfq written"
    h, w2 = C.fp4_contiguous_ref(case)
    assert np.array_equal(w2, written)
    q_ref, sf_ref = S.swiglu_quantize(h[written])
    C.compare_quantised(qh[written], sf_bytes[written], q_ref, sf_ref, _y_ref(h[written]), "fp4 contiguous swiglu")
    q_o, sf_o, _ = FP4.m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(case["a"], case["sfa"], case["b"], case["sfb"],
                                                                  case["m_indices"])
    assert np.array_equal(q_o[written], q_ref) and np.array_equal(sf_o[written], sf_ref)


def test_fp4_masked_swiglu_parity(fg):
    from gpu_util import dev
    inter = 384
    masks = [0, 1, 129, 200, 64, 33]
    case = C.fp4_masked_case(32, num_groups=len(masks), m_max=200, n=2 * inter, k=256, masked_m=masks)
    g_, m_max = case["g"], case["m_max"]
    q = torch.full((g_, m_max, inter), SENT_Q, dtype=torch.uint8, device="cuda")
    sfq = torch.full((g_, (inter + 511) // 512, (m_max + 3) // 4 * 4), SENT_W, dtype=torch.int32, device="cuda")
    fg.m_grouped_fp8_fp4_gemm_nt_masked_swiglu(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                               dev(case["masked_m"]), q, sfq)
    _status_ok(fg)
    qh, sfh = q.cpu().numpy(), sfq.cpu().numpy()
    ref = FP4.m_grouped_fp8_fp4_gemm_nt_masked_swiglu(case["a"], case["sfa"], case["b"], case["sfb"],
                                                     case["masked_m"])
    hs = C.fp4_masked_ref(case)
    for e in range(g_):
        mm = int(case["masked_m"][e])
        assert np.all(qh[e, mm:] == SENT_Q), f"group {e}: rows beyond the mask written"
        sb = F.unpack_ue8m0(sfh[e], m_max, inter // 128)
        sent = F.unpack_ue8m0(np.full_like(sfh[e], SENT_W), m_max, inter // 128)
        assert np.array_equal(sb[mm:], sent[mm:]), f"group {e}: scale bytes beyond the mask written"
        if mm:
            C.compare_quantised(qh[e, :mm], sb[:mm], ref[e][0], ref[e][1], _y_ref(hs[e]),
                                f"fp4 masked swiglu group {e}")


def test_fp4_swiglu_exact_probe_bit_exact(fg):
    """A[m, 0] in {1, 2}, the rest 0; gate row i has one code g_i in {4, 6} (scale 2^4: 64
    or 96), up row i one code in {-2, -1, 0, 1, 2, 3}: the GEMM is exact and SiLU(gate) ==
    gate in FP32 and FP64 (gate >= 64), so codes and scales must be identical."""
    from gpu_util import dev
    g = np.random.Generator(np.random.PCG64(33))
    inter, k, m_total = 256, 128, 256
    a = np.zeros((m_total, k), np.uint8)
    a[:, 0] = np.where(g.integers(0, 2, m_total) == 0, 0x38, 0x40)
    codes = np.zeros((1, 2 * inter, k), np.uint8)
    codes[0, :inter, 0] = np.array([0x6, 0x7], np.uint8)[g.integers(0, 2, inter)]            # 4, 6
    codes[0, inter:, 0] = np.array([0xC, 0xA, 0x0, 0x2, 0x4, 0x5], np.uint8)[g.integers(0, 6, inter)]
    b = FP4.pack_fp4(codes)
    sb = np.full((2 * inter, k // 32), 127, np.uint8)
    sb[:inter, 0] = 131                                                                        # gate x 16
    sfa = F.pack_ue8m0(np.full((m_total, 1), 127, np.uint8))
    sfb = FP4.pack_mx_scales(sb)[None]
    m_indices = np.zeros(m_total, np.int32)
    q = torch.full((m_total, inter), SENT_Q, dtype=torch.uint8, device="cuda")
    sfq = torch.zeros((1, (m_total + 3) // 4 * 4), dtype=torch.int32, device="cuda")
    fg.m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(dev(a), dev(sfa), dev(b), dev(sfb), dev(m_indices), q, sfq)
    _status_ok(fg)
    q_ref, sf_ref, _ = FP4.m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(a, sfa, b, sfb, m_indices)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(F.unpack_ue8m0(sfq.cpu().numpy(), m_total, inter // 128), sf_ref)


def test_fp4_moe_expert_chain(fg):
    """The Mega MoE expert computation in FP8 x FP4 on one GPU: linear 1 (gate-up, FP4
    weights) with the fused SwiGLU + E4M3 requantisation, its output consumed as is by
    linear 2 (the down projection, FP4 weights).  Linear 1's codes are checked against the
    oracle's, and linear 2 against the oracle GEMM on the codes linear 1 produced."""
    from gpu_util import GuardedOut, dev
    from oracle import swiglu as S
    inter, hidden = 256, 384
    case = C.fp4_contiguous_case(35, num_tokens=256, num_routed=8, topk=2, num_groups=3, n=2 * inter, k=256)
    m_total = case["m_total"]
    q = torch.zeros((m_total, inter), dtype=torch.uint8, device="cuda")
    sfq = torch.zeros(((inter + 511) // 512, (m_total + 3) // 4 * 4), dtype=torch.int32, device="cuda")
    fg.m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(dev(case["a"]), dev(case["sfa"]), dev(case["b"]),
                                                   dev(case["sfb"]), dev(case["m_indices"]), q, sfq)
    _status_ok(fg)
    written = case["m_indices"] >= 0
    h, _ = C.fp4_contiguous_ref(case)
    q_ref, sf_ref = S.swiglu_quantize(h[written])
    qh, sfh = q.cpu().numpy(), sfq.cpu().numpy()
    C.compare_quantised(qh[written], F.unpack_ue8m0(sfh, m_total, inter // 128)[written], q_ref, sf_ref,
                        _y_ref(h[written]), "fp4 linear 1")
    gw = np.random.Generator(np.random.PCG64(36))
    w2, sfw2 = C._mxfp4_experts(gw.standard_normal((3, hidden, inter)) * 0.05)
    d = GuardedOut(m_total, hidden, "bf16")
    fg.m_grouped_fp8_fp4_gemm_nt_contiguous(q, sfq, dev(w2), dev(sfw2), dev(case["m_indices"]), d.tensor)
    _status_ok(fg)
    d.check_guards()
    ref, _ = FP4.m_grouped_fp8_fp4_gemm_nt_contiguous(qh, sfh, w2, sfw2, case["m_indices"])
    assert np.array_equal(~d.is_sentinel(), written)
    C.compare(d.values()[written], ref[written], "fp4 linear 2 on linear 1's output")


@pytest.mark.parametrize("split", ["2", "4"])
def test_fp4_scale_selection_probe_split_k(fg, split, monkeypatch, capfd):
    """The bit-exact scale probe under split-K clusters: each CTA's share of the 6 K-groups
    starts at its own K-group (uneven shares at 4), so both the A word (four K-groups) and
    the B word (one K-group) of its first stage come from mid-array; partial sums of powers
    of two stay exact."""
    from gpu_util import GuardedOut, dev
    monkeypatch.setenv("FG_FORCE_SPLIT", split)
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    m, n, k = 64, 384, 768
    sa = (126 + (np.arange(m)[:, None] + np.arange(k // 128)[None, :]) % 3).astype(np.uint8)
    sb = (124 + (np.arange(n)[:, None] + 3 * np.arange(k // 32)[None, :]) % 7).astype(np.uint8)
    a = np.full((m, k), 0x38, np.uint8)
    b = np.full((n, k // 2), 0x22, np.uint8)
    out = GuardedOut(m, n, "f32")
    fg.fp8_fp4_gemm_nt(dev(a), dev(F.pack_ue8m0(sa)), dev(b), dev(FP4.pack_mx_scales(sb)), out.tensor)
    _status_ok(fg)
    assert _launched(capfd, "fp8_fp4_gemm_nt")["split"] == split
    want = 32.0 * (np.repeat(np.exp2(sa - 127.0), 4, axis=1) @ np.exp2(sb - 127.0).T)
    assert np.array_equal(out.values(), want)


def test_fp4_contiguous_empty_groups_and_all_padding_block(fg):
    """Expert 1 receives no tokens and the last block is all padding: with FP4 weights the
    written rows and their values match the oracle and nothing else is written."""
    from gpu_util import GuardedOut, dev
    import oracle_pins as P
    g = np.random.Generator(np.random.PCG64(37))
    m_indices = np.array([0] * 130 + [-1] * 126 + [2] * 128 + [-1] * 128, np.int32)
    k, n, groups = 256, 128, 3
    a = P.rand_codes(g, (len(m_indices), k))
    b = P.rand_fp4(g, (groups, n, k // 2))
    sfa = P.rand_words(g, len(m_indices), k // 128)
    sfb = np.stack([P.rand_words(g, n, k // 32) for _ in range(groups)])
    d = GuardedOut(len(m_indices), n, "bf16")
    fg.m_grouped_fp8_fp4_gemm_nt_contiguous(dev(a), dev(sfa), dev(b), dev(sfb), dev(m_indices), d.tensor)
    _status_ok(fg)
    d.check_guards()
    ref, written = FP4.m_grouped_fp8_fp4_gemm_nt_contiguous(a, sfa, b, sfb, m_indices)
    assert np.array_equal(~d.is_sentinel(), written)
    C.compare(d.values()[written], ref[written], "fp4 contiguous edge")
