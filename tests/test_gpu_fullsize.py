"""GPU parity at the full benchmark sizes, in the launch configuration bench.py times
(default tile choice, all SMs).  The oracle computes sampled output rows one by one;
every row that must stay untouched is checked bit-exactly, and every output is checked
finite."""
import numpy as np
import pytest

import cases as C

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_fp8_e4m3_gb300 as lib
    return lib


def _ok(fg):
    st, detail = fg.get_device_error()
    assert st == 0, (st, hex(detail))


def _rows(m, n_samples, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    r = set(g.choice(m, size=min(m, n_samples), replace=False).tolist())
    r |= {0, m - 1, min(127, m - 1), min(128, m - 1)}
    return np.array(sorted(r))


@pytest.mark.parametrize("m,n,k", [(4096, 7168, 2048), (64, 7168, 4096)])
def test_dense_pair_full_size(fg, m, n, k):
    from gpu_util import GuardedOut, dev
    case = C.dense_case(1001, m, n, k, True, "f32")
    out = GuardedOut(m, n, "f32")
    fg.fp8_gemm_nt(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]), out.tensor,
                   c=dev(case["c"]))
    _ok(fg)
    out.check_guards()
    got = out.values()
    assert np.all(np.isfinite(got))
    rows = _rows(m, 48, 5)
    C.compare(got[rows], C.dense_ref(case, rows=rows), f"dense {m}x{n}x{k} sampled rows")


def test_contiguous_full_size(fg):
    from gpu_util import GuardedOut, dev
    case = C.contiguous_case(1002)            # 8192 tokens, top-6 of 256, experts 0-31, N=K=4096
    d = GuardedOut(case["m_total"], case["n"], "bf16")
    fg.m_grouped_fp8_gemm_nt_contiguous(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                        dev(case["m_indices"]), d.tensor)
    _ok(fg)
    d.check_guards()
    written = case["m_indices"] >= 0
    assert np.array_equal(~d.is_sentinel(), written), "padding rows written or valid rows missing"
    vals = d.values()
    assert np.all(np.isfinite(vals[written]))
    valid_rows = np.nonzero(written)[0]
    g = np.random.Generator(np.random.PCG64(6))
    rows = np.sort(g.choice(valid_rows, size=48, replace=False))
    ref, _ = C.contiguous_ref(case, rows=rows)
    C.compare(vals[rows], ref, "contiguous sampled rows")


def test_masked_full_size(fg):
    from gpu_util import GuardedOut, dev
    case = C.masked_case(1003)                # 32 experts x 256 rows, N=4096, K=2048
    g_, m_max, n = case["g"], case["m_max"], case["n"]
    d = GuardedOut(g_ * m_max, n, "bf16")
    fg.m_grouped_fp8_gemm_nt_masked(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                    dev(case["masked_m"]), d.tensor.view(g_, m_max, n),
                                    expected_m=int(np.mean(case["masked_m"])))
    _ok(fg)
    d.check_guards()
    sent = d.is_sentinel().reshape(g_, m_max)
    vals = d.values().reshape(g_, m_max, n)
    for e in range(g_):
        mm = int(case["masked_m"][e])
        assert not sent[e, :mm].any() and sent[e, mm:].all(), f"group {e}: rows beyond the mask written"
        assert np.all(np.isfinite(vals[e, :mm]))
    # sampled rows of every expert: the first and last valid row and up to six more
    g = np.random.Generator(np.random.PCG64(11))
    rows = {}
    for e in range(g_):
        mm = int(case["masked_m"][e])
        pick = set(g.choice(mm, size=min(mm, 6), replace=False).tolist()) if mm > 0 else set()
        rows[e] = np.array(sorted(pick | ({0, mm - 1} if mm > 0 else set())), dtype=np.int64)
    ref = C.masked_ref(case, rows=rows)
    for e in range(g_):
        C.compare(vals[e, rows[e]], ref[e], f"masked group {e} sampled rows")


@pytest.mark.parametrize("alias", [False, True])
def test_k_grouped_full_size(fg, alias):
    from gpu_util import GuardedOut, dev
    case = C.k_grouped_case(1004)             # 8 experts, M=4096, N=2048, sum K = 16384 (padded)
    g_, m, n = case["g"], case["m"], case["n"]
    d = GuardedOut(g_ * m, n, "f32")
    if alias:
        d.fill_from(case["c"].reshape(g_ * m, n))
        c_t = d.tensor.view(g_, m, n)
    else:
        c_t = dev(case["c"])
    fg.k_grouped_fp8_gemm_tn_contiguous(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                        dev(case["ks"]), d.tensor.view(g_, m, n), c=c_t)
    _ok(fg)
    d.check_guards()
    vals = d.values().reshape(g_, m, n)
    assert np.all(np.isfinite(vals))
    rows = _rows(m, 12, 7)
    ref = C.k_grouped_ref(case, rows=rows)
    for e in range(g_):
        C.compare(vals[e][rows], ref[e], f"k-grouped group {e} sampled rows")


def test_contiguous_swiglu_full_size(fg):
    """The fused gate-up GEMM at the contiguous benchmark shape read as gate + up
    (8192 tokens, top-6 of 256, experts 0-31, B [32, 2 x 2048, 4096]): sampled valid rows
    against the oracle, every padding row untouched."""
    from gpu_util import dev
    from oracle import swiglu as S
    from test_gpu_swiglu import SENT_Q, _sf_bytes, _y_ref, compare_quantised
    case = C.contiguous_case(1005)
    m_total, inter = case["m_total"], case["n"] // 2
    q = torch.full((m_total, inter), SENT_Q, dtype=torch.uint8, device="cuda")
    sfq = torch.zeros(((inter + 511) // 512, (m_total + 3) // 4 * 4), dtype=torch.int32, device="cuda")
    fg.m_grouped_fp8_gemm_nt_contiguous_swiglu(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                               dev(case["m_indices"]), q, sfq)
    _ok(fg)
    qh = q.cpu().numpy()
    written = case["m_indices"] >= 0
    assert np.all(qh[~written] == SENT_Q), "padding rows written"
    g = np.random.Generator(np.random.PCG64(8))
    rows = np.sort(g.choice(np.nonzero(written)[0], size=48, replace=False))
    h, _ = C.contiguous_ref(case, rows=rows)
    q_ref, sf_ref = S.swiglu_quantize(h)
    sf = _sf_bytes(sfq.cpu().numpy(), m_total, inter // 128)[rows]
    compare_quantised(qh[rows], sf, q_ref, sf_ref, _y_ref(h), "contiguous swiglu full size")


def test_mqa_logits_full_size(fg):
    """Causal MQA logits at the benchmark size (4096 query x 4096 kv tokens, 64 heads,
    D = 128): sampled query rows against the oracle, -inf above the diagonal."""
    from test_gpu_mqa import check, mqa_case, run
    case = mqa_case(1006, 4096, 4096, "causal")
    got = run(fg, case, True)
    rows = _rows(4096, 24, 9)
    check(case, got, True, rows=rows)


# ------------------------------------------------------------------ FP8 x FP4
def test_fp4_prefill_full_size(fg):
    """The FP8 x FP4 prefill 4096 x 7168 x 2048 with FP32 C (MXFP4 weights); the decode shape
    is compared in full by the FP4 parity tests."""
    from gpu_util import GuardedOut, dev
    m, n, k = 4096, 7168, 2048
    case = C.fp4_dense_case(1011, m, n, k, True, "f32")
    out = GuardedOut(m, n, "f32")
    fg.fp8_fp4_gemm_nt(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]), out.tensor,
                       c=dev(case["c"]))
    _ok(fg)
    out.check_guards()
    got = out.values()
    assert np.all(np.isfinite(got))
    rows = _rows(m, 48, 12)
    C.compare(got[rows], C.fp4_dense_ref(case, rows=rows), "fp4 prefill sampled rows")


def test_fp4_contiguous_full_size(fg):
    from gpu_util import GuardedOut, dev
    case = C.fp4_contiguous_case(1012)        # 8192 tokens, top-6 of 256, experts 0-31, N=K=4096
    d = GuardedOut(case["m_total"], case["n"], "bf16")
    fg.m_grouped_fp8_fp4_gemm_nt_contiguous(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                            dev(case["m_indices"]), d.tensor)
    _ok(fg)
    d.check_guards()
    written = case["m_indices"] >= 0
    assert np.array_equal(~d.is_sentinel(), written), "padding rows written or valid rows missing"
    vals = d.values()
    assert np.all(np.isfinite(vals[written]))
    g = np.random.Generator(np.random.PCG64(13))
    rows = np.sort(g.choice(np.nonzero(written)[0], size=48, replace=False))
    ref, _ = C.fp4_contiguous_ref(case, rows=rows)
    C.compare(vals[rows], ref, "fp4 contiguous sampled rows")


def test_fp4_masked_full_size(fg):
    from gpu_util import GuardedOut, dev
    case = C.fp4_masked_case(1013)            # 32 experts x 256 rows, N=4096, K=2048
    g_, m_max, n = case["g"], case["m_max"], case["n"]
    d = GuardedOut(g_ * m_max, n, "bf16")
    fg.m_grouped_fp8_fp4_gemm_nt_masked(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]),
                                        dev(case["masked_m"]), d.tensor.view(g_, m_max, n),
                                        expected_m=int(np.mean(case["masked_m"])))
    _ok(fg)
    d.check_guards()
    sent = d.is_sentinel().reshape(g_, m_max)
    vals = d.values().reshape(g_, m_max, n)
    g = np.random.Generator(np.random.PCG64(14))
    rows = {}
    for e in range(g_):
        mm = int(case["masked_m"][e])
        assert not sent[e, :mm].any() and sent[e, mm:].all(), f"group {e}: rows beyond the mask written"
        assert np.all(np.isfinite(vals[e, :mm]))
        pick = set(g.choice(mm, size=min(mm, 6), replace=False).tolist()) if mm > 0 else set()
        rows[e] = np.array(sorted(pick | ({0, mm - 1} if mm > 0 else set())), dtype=np.int64)
    ref = C.fp4_masked_ref(case, rows=rows)
    for e in range(g_):
        C.compare(vals[e, rows[e]], ref[e], f"fp4 masked group {e} sampled rows")


def test_fp4_contiguous_swiglu_full_size(fg):
    """The fused gate-up GEMM with FP4 weights at the contiguous benchmark shape
    (B [32, 2 x 2048, 4096] packed E2M1): sampled valid rows, every padding row untouched."""
    from gpu_util import dev
    from oracle import swiglu as S
    from test_gpu_swiglu import SENT_Q, _sf_bytes, _y_ref, compare_quantised
    case = C.fp4_contiguous_case(1014)
    m_total, inter = case["m_total"], case["n"] // 2
    q = torch.full((m_total, inter), SENT_Q, dtype=torch.uint8, device="cuda")
    sfq = torch.zeros(((inter + 511) // 512, (m_total + 3) // 4 * 4), dtype=torch.int32, device="cuda")
    fg.m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(dev(case["a"]), dev(case["sfa"]), dev(case["b"]),
                                                   dev(case["sfb"]), dev(case["m_indices"]), q, sfq)
    _ok(fg)
    qh = q.cpu().numpy()
    written = case["m_indices"] >= 0
    assert np.all(qh[~written] == SENT_Q), "padding rows written"
    g = np.random.Generator(np.random.PCG64(15))
    rows = np.sort(g.choice(np.nonzero(written)[0], size=48, replace=False))
    h, _ = C.fp4_contiguous_ref(case, rows=rows)
    q_ref, sf_ref = S.swiglu_quantize(h)
    sf = _sf_bytes(sfq.cpu().numpy(), m_total, inter // 128)[rows]
    compare_quantised(qh[rows], sf, q_ref, sf_ref, _y_ref(h), "fp4 contiguous swiglu full size")


@pytest.mark.parametrize("weights", ["fp8", "fp4"])
def test_masked_swiglu_full_size(fg, weights):
    """The fused gate-up GEMM in the masked layout at the masked benchmark shape read as gate
    + up (32 experts x 256 rows, B [32, 2 x 2048, 2048]): sampled rows of every expert
    against the oracle, rows past each mask untouched."""
    from gpu_util import dev
    from oracle import fp4 as FP4
    from oracle import swiglu as S
    from test_gpu_swiglu import SENT_Q, _sf_bytes, _y_ref, compare_quantised
    case = C.masked_case(1015, weights=weights)
    g_, m_max, inter = case["g"], case["m_max"], case["n"] // 2
    q = torch.full((g_, m_max, inter), SENT_Q, dtype=torch.uint8, device="cuda")
    sfq = torch.zeros((g_, (inter + 511) // 512, (m_max + 3) // 4 * 4), dtype=torch.int32, device="cuda")
    call = fg.m_grouped_fp8_fp4_gemm_nt_masked_swiglu if weights == "fp4" else fg.m_grouped_fp8_gemm_nt_masked_swiglu
    call(dev(case["a"]), dev(case["sfa"]), dev(case["b"]), dev(case["sfb"]), dev(case["masked_m"]), q, sfq)
    _ok(fg)
    qh, sfh = q.cpu().numpy(), sfq.cpu().numpy()
    g = np.random.Generator(np.random.PCG64(16))
    rows = {}
    for e in range(g_):
        mm = int(case["masked_m"][e])
        assert np.all(qh[e, mm:] == SENT_Q), f"group {e}: rows beyond the mask written"
        pick = set(g.choice(mm, size=min(mm, 4), replace=False).tolist()) if mm > 0 else set()
        rows[e] = np.array(sorted(pick | ({0, mm - 1} if mm > 0 else set())), dtype=np.int64)
    ref_gemm = FP4.m_grouped_fp8_fp4_gemm_nt_masked if weights == "fp4" else C.oracle.m_grouped_fp8_gemm_nt_masked
    hs = ref_gemm(case["a"], case["sfa"], case["b"], case["sfb"], case["masked_m"], rows=rows)
    for e in range(g_):
        if len(rows[e]) == 0:
            continue
        q_ref, sf_ref = S.swiglu_quantize(hs[e])
        sf = _sf_bytes(sfh[e], m_max, inter // 128)[rows[e]]
        compare_quantised(qh[e, rows[e]], sf, q_ref, sf_ref, _y_ref(hs[e]), f"masked swiglu {weights} group {e}")
