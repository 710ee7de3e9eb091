"""GPU parity of the gate-up GEMM with the fused SwiGLU + per-1x128 FP8 requantisation.

The kernel evaluates SiLU(gate) * up in FP32 from FP32 accumulators and quantises those
FP32 values; the oracle evaluates the GEMM and SwiGLU in FP64 and quantises the value
rounded to FP32.  Upstream rounding therefore moves a value across an E4M3 rounding
boundary (one code apart) or a group's amax across a power of two (one scale apart) only
where the two results sit within ~1e-6 of such a boundary.  The checks: every dequantised
output within one E4M3 spacing (2^-3 relative, 2^-9 of the scale below the normal range)
plus the upstream error of the oracle's dequantised value, at least 99% of codes and scale
bytes identical, a bit-exact probe where no rounding happens upstream (gate >= 64 makes
SiLU(gate) == gate in both precisions), and rows that must stay untouched bit-exact."""
import numpy as np
import pytest

import cases as C
from oracle import formats as F
from oracle import swiglu as S

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SENT_Q = 0xAB
SENT_W = -0x21436588          # 0xDEBC9A78 as int32


@pytest.fixture(scope="module")
def fg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_fp8_e4m3_gb300 as lib
    return lib


def _ok(fg):
    st, detail = fg.get_device_error()
    assert st == 0, (st, hex(detail))


compare_quantised = C.compare_quantised


def _sf_bytes(words, rows, groups):
    """packed words [ceil(groups/4)][>= rows] -> bytes [rows, groups]"""
    return F.unpack_ue8m0(words, rows, groups)


def _y_ref(h):
    return S.swiglu(h).astype(np.float32).astype(np.float64)


def test_contiguous_swiglu_parity(fg):
    from gpu_util import dev
    inter = 256
    case = C.contiguous_case(21, num_tokens=512, num_routed=16, topk=3, num_groups=5, n=2 * inter, k=384)
    m_total = case["m_total"]
    q = torch.full((m_total, inter), SENT_Q, dtype=torch.uint8, device="cuda")
    sfq = torch.full(((inter + 511) // 512, (m_total + 3) // 4 * 4), SENT_W, dtype=torch.int32, device="cuda")
    fg.m_grouped_fp8_gemm_nt_contiguous_swiglu(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                               dev(case["m_indices"]), q, sfq)
    _ok(fg)
    qh, sfh = q.cpu().numpy(), sfq.cpu().numpy()
    written = case["m_indices"] >= 0
    assert np.all(qh[~written] == SENT_Q), "padding rows of q written"
    sf_bytes = _sf_bytes(sfh, m_total, inter // 128)
    sent_bytes = _sf_bytes(np.full_like(sfh, SENT_W), m_total, inter // 128)
    assert np.array_equal(sf_bytes[~written], sent_bytes[~written]), "padding rows of sfq written"
    h, w2 = C.contiguous_ref(case)
    assert np.array_equal(w2, written)
    q_ref, sf_ref = S.swiglu_quantize(h[written])
    compare_quantised(qh[written], sf_bytes[written], q_ref, sf_ref, _y_ref(h[written]), "contiguous swiglu")


def test_masked_swiglu_parity(fg):
    from gpu_util import dev
    inter = 384
    case = C.masked_case(22, num_groups=6, m_max=200, n=2 * inter, k=256)
    g_, m_max = case["g"], case["m_max"]
    q = torch.full((g_, m_max, inter), SENT_Q, dtype=torch.uint8, device="cuda")
    sfq = torch.full((g_, (inter + 511) // 512, (m_max + 3) // 4 * 4), SENT_W, dtype=torch.int32, device="cuda")
    fg.m_grouped_fp8_gemm_nt_masked_swiglu(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                           dev(case["masked_m"]), q, sfq)
    _ok(fg)
    qh, sfh = q.cpu().numpy(), sfq.cpu().numpy()
    ref = S.m_grouped_fp8_gemm_nt_masked_swiglu(case["a"], case["sfa"], case["b"], case["sfb"], case["masked_m"])
    hs = C.masked_ref(case)
    for e in range(g_):
        mm = int(case["masked_m"][e])
        assert np.all(qh[e, mm:] == SENT_Q), f"group {e}: rows beyond the mask written"
        sb = _sf_bytes(sfh[e], m_max, inter // 128)
        sent = _sf_bytes(np.full_like(sfh[e], SENT_W), m_max, inter // 128)
        assert np.array_equal(sb[mm:], sent[mm:]), f"group {e}: scale bytes beyond the mask written"
        if mm:
            compare_quantised(qh[e, :mm], sb[:mm], ref[e][0], ref[e][1], _y_ref(hs[e]), f"masked swiglu group {e}")


def test_swiglu_exact_probe_bit_exact(fg):
    """A[m, 0] = a_m in {1, 2}, the rest 0; gate row i has one entry g_i in [64, 120], up row
    i one entry u_i in [-3, 3]: h is exact, SiLU(gate) == gate in FP32 and FP64, so
    y = a_m^2 g_i u_i exactly and codes and scales must be identical."""
    from gpu_util import dev
    g = np.random.Generator(np.random.PCG64(23))
    inter, k, m_total = 256, 128, 256
    codes_g = np.arange(0x68, 0x70, dtype=np.uint8)                                  # 64, 72, .., 120
    codes_u = np.array([0xC0, 0xB8, 0x00, 0x38, 0x40, 0x44], np.uint8)              # -2,-1,0,1,2,3
    a = np.zeros((m_total, k), np.uint8)
    a[:, 0] = np.where(g.integers(0, 2, m_total) == 0, 0x38, 0x40)                   # 1 or 2
    b = np.zeros((1, 2 * inter, k), np.uint8)
    b[0, :inter, 0] = codes_g[g.integers(0, len(codes_g), inter)]
    b[0, inter:, 0] = codes_u[g.integers(0, len(codes_u), inter)]
    sfa = F.pack_ue8m0(np.full((m_total, 1), 127, np.uint8))
    sfb = F.pack_ue8m0(np.full((2 * inter // 128, 1), 127, np.uint8))[None]
    m_indices = np.zeros(m_total, np.int32)
    q = torch.full((m_total, inter), SENT_Q, dtype=torch.uint8, device="cuda")
    sfq = torch.zeros((1, (m_total + 3) // 4 * 4), dtype=torch.int32, device="cuda")
    fg.m_grouped_fp8_gemm_nt_contiguous_swiglu(dev(a), dev(sfa), dev(b), dev(sfb), dev(m_indices), q, sfq)
    _ok(fg)
    q_ref, sf_ref, _ = S.m_grouped_fp8_gemm_nt_contiguous_swiglu(a, sfa, b, sfb, m_indices)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(_sf_bytes(sfq.cpu().numpy(), m_total, inter // 128), sf_ref)


def test_contiguous_swiglu_feeds_down_projection(fg):
    """The quantised output is consumed as is by the down-projection GEMM (same layout as
    an activation quantised by the library's row quantiser)."""
    from gpu_util import GuardedOut, dev
    inter, hidden = 256, 384
    case = C.contiguous_case(24, num_tokens=256, num_routed=8, topk=2, num_groups=3, n=2 * inter, k=256)
    m_total = case["m_total"]
    q = torch.zeros((m_total, inter), dtype=torch.uint8, device="cuda")
    sfq = torch.zeros(((inter + 511) // 512, (m_total + 3) // 4 * 4), dtype=torch.int32, device="cuda")
    fg.m_grouped_fp8_gemm_nt_contiguous_swiglu(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                               dev(case["m_indices"]), q, sfq)
    gw = np.random.Generator(np.random.PCG64(25))
    w2 = np.empty((3, hidden, inter), np.uint8)
    sfw2 = []
    for e in range(3):
        w2[e], sb = F.quantize_blocks(gw.standard_normal((hidden, inter)) * 0.05)
        sfw2.append(F.pack_ue8m0(sb))
    sfw2 = np.stack(sfw2)
    d = GuardedOut(m_total, hidden, "bf16")
    fg.m_grouped_fp8_gemm_nt_contiguous(q, sfq, dev(w2), dev(sfw2), dev(case["m_indices"]), d.tensor)
    _ok(fg)
    written = case["m_indices"] >= 0
    ref, _ = C.oracle.m_grouped_fp8_gemm_nt_contiguous(q.cpu().numpy(), sfq.cpu().numpy(), w2, sfw2,
                                                      case["m_indices"])
    C.compare(d.values()[written], ref[written], "down projection of the fused output")
