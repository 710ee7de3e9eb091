"""GPU parity of long accumulations: the promotion step of the fine-grained FP8 GEMM.

The article "Deepseek AI Libera DeepGEMM" ("Details and technical benefits") gives the
reason for fine-grained scaling with promotion: FP8 tensor-core accumulation is
imprecise, so partial sums are promoted to FP32 with their scales applied.  Here the
block-scaled MMA applies the UE8M0 scales inside the tensor core and accumulates in FP32
tensor memory over the whole K loop.  These tests check that reading at K = 16384 with
per-group magnitudes spanning about +-20 binades, falling along K so that the smallest
groups are added after the largest, in every launch form the dense GEMM can take (one
CTA per tile, split-K clusters), in the K-grouped GEMM with one expert owning all of K, and
at the decode shape (M = 64)."""
import numpy as np
import pytest

import cases as C
import oracle
import workloads
from oracle import formats as F

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

K_LONG = 16384


@pytest.fixture(scope="module")
def fg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_fp8_e4m3_gb300 as lib
    return lib


def _ok(fg):
    st, detail = fg.get_device_error()
    assert st == 0, (st, hex(detail))


def wide_dense_case(seed, m, n, k, with_c, out):
    w = workloads.dense_wide_range(seed, m, n, k, with_c)
    a, sa = F.quantize_rows(w["a"])
    b, sb = F.quantize_blocks(w["b"])
    assert int(sa.max()) - int(sa.min()) >= 18 and int(sb.max()) - int(sb.min()) >= 18
    return {"m": m, "n": n, "k": k, "a": a, "sfa": F.pack_ue8m0(sa), "b": b, "sfb": F.pack_ue8m0(sb),
            "c": w["c"], "out": out}


@pytest.mark.parametrize("form", ["default", "one_cta", "split4"])
@pytest.mark.parametrize("with_c,out", [(True, "f32"), (False, "f32"), (False, "bf16")])
def test_dense_k16384_wide_range(fg, form, with_c, out, monkeypatch):
    from gpu_util import GuardedOut, dev
    m, n, k = 256, 512, K_LONG
    if form == "one_cta":
        monkeypatch.setenv("FG_FORCE_SPLIT", "1")
    elif form == "split4":
        monkeypatch.setenv("FG_FORCE_SPLIT", "4")
    case = wide_dense_case(4242, m, n, k, with_c, out)
    got = GuardedOut(m, n, out)
    c_t = dev(case["c"]) if with_c else None
    fg.fp8_gemm_nt(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]), got.tensor, c=c_t)
    _ok(fg)
    got.check_guards()
    ref = oracle.fp8_gemm_nt(case["a"], case["sfa"], case["b"], case["sfb"], case["c"])
    C.compare(got.values(), ref, f"dense {m}x{n}x{k} wide-range scales ({form})")


@pytest.mark.parametrize("m", [64, 1])
def test_decode_shape_k16384_wide_range(fg, m):
    """The decode shape (few rows, many weight columns) at K = 16384."""
    from gpu_util import GuardedOut, dev
    n, k = 1024, K_LONG
    case = wide_dense_case(4243 + m, m, n, k, True, "f32")
    got = GuardedOut(m, n, "f32")
    fg.fp8_gemm_nt(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]), got.tensor,
                   c=dev(case["c"]))
    _ok(fg)
    got.check_guards()
    ref = oracle.fp8_gemm_nt(case["a"], case["sfa"], case["b"], case["sfb"], case["c"])
    C.compare(got.values(), ref, f"dense {m}x{n}x{k} wide-range scales")


@pytest.mark.parametrize("alias", [False, True])
def test_k_grouped_single_expert_owns_k(fg, alias):
    """ks = [16384, 0, 0, 0]: expert 0 accumulates over all of K; experts 1-3 get D = C."""
    from gpu_util import GuardedOut, dev
    ks = [K_LONG, 0, 0, 0]
    g_, m, n = len(ks), 256, 256
    w = workloads.k_grouped_wide_range(4244, ks, m, n)
    a, sa = F.quantize_cols(w["a"])
    b, sb = F.quantize_cols(w["b"])
    sfa, sfb = F.pack_ue8m0(sa), F.pack_ue8m0(sb)
    d = GuardedOut(g_ * m, n, "f32")
    if alias:
        d.fill_from(w["c"].reshape(g_ * m, n))
        c_t = d.tensor.view(g_, m, n)
    else:
        c_t = dev(w["c"])
    fg.k_grouped_fp8_gemm_tn_contiguous(dev(a), dev(sfa), dev(b), dev(sfb), dev(w["ks"]),
                                        d.tensor.view(g_, m, n), c=c_t)
    _ok(fg)
    d.check_guards()
    vals = d.values().reshape(g_, m, n)
    ref = oracle.k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, w["ks"], w["c"])
    C.compare(vals[0], ref[0], "k-grouped expert 0, K = 16384, wide-range scales")
    for e in range(1, g_):
        assert np.array_equal(vals[e].astype(np.float32), w["c"][e]), f"expert {e}: D != C"


# ------------------------------------------------------------------ FP8 x FP4
def wide_fp4_case(seed, m, n, k, with_c, out):
    """The wide-range draws with the weights quantised to MXFP4 (E2M1, one scale per 32 K
    elements of a row), so B's scales vary per row and 32-wide block as well."""
    from oracle import fp4 as FP4
    w = workloads.dense_wide_range(seed, m, n, k, with_c)
    a, sa = F.quantize_rows(w["a"])
    b, sb = FP4.quantize_mxfp4(w["b"])
    assert int(sa.max()) - int(sa.min()) >= 18 and int(sb.max()) - int(sb.min()) >= 18
    return {"m": m, "n": n, "k": k, "a": a, "sfa": F.pack_ue8m0(sa), "b": b, "sfb": FP4.pack_mx_scales(sb),
            "c": w["c"], "out": out}


@pytest.mark.parametrize("form", ["default", "one_cta", "split4"])
@pytest.mark.parametrize("m,n", [(256, 512), (64, 1024)])
def test_fp4_k16384_wide_range(fg, form, m, n, monkeypatch):
    """The FP8 x FP4 GEMM at K = 16384 with falling wide-range magnitudes: the scales of both
    operands are applied per 32-wide K step inside the tensor core and the FP32 accumulator
    holds the whole K loop, in every dense launch form."""
    from gpu_util import GuardedOut, dev
    if form == "one_cta":
        monkeypatch.setenv("FG_FORCE_SPLIT", "1")
    elif form == "split4":
        monkeypatch.setenv("FG_FORCE_SPLIT", "4")
    case = wide_fp4_case(4250 + m, m, n, K_LONG, True, "f32")
    got = GuardedOut(m, n, "f32")
    fg.fp8_fp4_gemm_nt(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]), got.tensor,
                       c=dev(case["c"]))
    _ok(fg)
    got.check_guards()
    ref = oracle.fp8_fp4_gemm_nt(case["a"], case["sfa"], case["b"], case["sfb"], case["c"])
    C.compare(got.values(), ref, f"fp4 {m}x{n}x{K_LONG} wide-range scales ({form})")
