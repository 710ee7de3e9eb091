"""The tile choices of the benchmark shapes on a 152-SM GB300.

The host cost model picks the N tile (and, for dense GEMMs with few tiles, a split-K
cluster) per call.  These choices carry much of the measured performance (for instance
BN=224 with two TMEM accumulators against BN=256 with one on the M-grouped GEMMs, and 192
against 224 on the prefill, where the model's costs tie and whole waves decide), so a
change to the model that moves them should be deliberate: each benchmark shape is launched
once with FG_PRINT_CONFIGS=1 (zero operands; only the printed choice is checked here, the
results are covered by the parity tests)."""
import re

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected choices are those of a 152-SM GB300")
    import moe_fp8_e4m3_gb300 as lib
    return lib


def _u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8, device="cuda")


def _i32(*shape):
    return torch.zeros(shape, dtype=torch.int32, device="cuda")


def _cdiv(a, b):
    return (a + b - 1) // b


def _a4(x):
    return (x + 3) // 4 * 4


def _printed(capfd, prefix):
    torch.cuda.synchronize()
    err = capfd.readouterr().err
    lines = [ln for ln in err.splitlines() if ln.startswith("[fg] " + prefix)]
    assert lines, err
    return dict(re.findall(r"(\w+)=(-?\d+)", lines[-1]))


def _dense(fg, m, n, k, with_c, out):
    a, sfa = _u8(m, k), _i32(_cdiv(k, 512), _a4(m))
    b, sfb = _u8(n, k), _i32(_cdiv(k, 512), _a4(_cdiv(n, 128)))
    d = torch.zeros((m, n), dtype=torch.float32 if out == "f32" else torch.bfloat16, device="cuda")
    c = torch.zeros((m, n), dtype=torch.float32, device="cuda") if with_c else None
    fg.fp8_gemm_nt(a, sfa, b, sfb, d, c=c)


@pytest.mark.parametrize("m,n,k,with_c,out,bn,split", [
    (4096, 7168, 2048, True, "f32", 192, 1),    # the prefill: 8 whole waves (224: 7, the last partial)
    (64, 7168, 4096, True, "f32", 128, 2),      # the decode: 2-CTA split-K clusters
    (128, 256, 512, False, "bf16", 64, 1),      # the small case: unsplit
])
def test_dense_choices(fg, capfd, monkeypatch, m, n, k, with_c, out, bn, split):
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    _dense(fg, m, n, k, with_c, out)
    cfg = _printed(capfd, "fp8_gemm_nt")
    assert (int(cfg["BN"]), int(cfg["split"])) == (bn, split), cfg


def test_contiguous_choice(fg, capfd, monkeypatch):
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    g, m_total, n, k = 32, 8192, 4096, 4096
    m_indices = (torch.arange(m_total, device="cuda", dtype=torch.int32) // 256).contiguous()
    d = torch.zeros((m_total, n), dtype=torch.bfloat16, device="cuda")
    fg.m_grouped_fp8_gemm_nt_contiguous(_u8(m_total, k), _i32(_cdiv(k, 512), _a4(m_total)), _u8(g, n, k),
                                        _i32(g, _cdiv(k, 512), _a4(_cdiv(n, 128))), m_indices, d)
    assert int(_printed(capfd, "m_grouped_nt_contiguous")["BN"]) == 224


def test_masked_choice(fg, capfd, monkeypatch):
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    g, m_max, n, k = 32, 256, 4096, 2048
    masked_m = torch.full((g,), 128, dtype=torch.int32, device="cuda")   # the mean row count the hint carries
    d = torch.zeros((g, m_max, n), dtype=torch.bfloat16, device="cuda")
    fg.m_grouped_fp8_gemm_nt_masked(_u8(g, m_max, k), _i32(g, _cdiv(k, 512), _a4(m_max)), _u8(g, n, k),
                                    _i32(g, _cdiv(k, 512), _a4(_cdiv(n, 128))), masked_m, d, expected_m=128)
    assert int(_printed(capfd, "m_grouped_masked")["BN"]) == 224


def test_k_grouped_choice(fg, capfd, monkeypatch):
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    g, m, n, k_total = 8, 4096, 2048, 16384
    ks = torch.full((g,), k_total // g, dtype=torch.int32, device="cuda")
    c = torch.zeros((g, m, n), dtype=torch.float32, device="cuda")
    fg.k_grouped_fp8_gemm_tn_contiguous(_u8(k_total, m), _i32(_cdiv(k_total, 512), _a4(m)), _u8(k_total, n),
                                        _i32(_cdiv(k_total, 512), _a4(n)), ks, c, c=c)
    assert int(_printed(capfd, "k_grouped_tn")["BN"]) == 128


def _fp4_dense(fg, m, n, k):
    a, sfa = _u8(m, k), _i32(_cdiv(k, 512), _a4(m))
    b, sfb = _u8(n, k // 2), _i32(k // 128, _a4(n))
    d = torch.zeros((m, n), dtype=torch.float32, device="cuda")
    fg.fp8_fp4_gemm_nt(a, sfa, b, sfb, d, c=torch.zeros((m, n), dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("m,n,k,bn,split", [
    (4096, 7168, 2048, 224, 1),    # the prefill shape with FP4 weights
    (64, 7168, 4096, 128, 2),      # the decode shape with FP4 weights
])
def test_fp4_dense_choices(fg, capfd, monkeypatch, m, n, k, bn, split):
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    _fp4_dense(fg, m, n, k)
    cfg = _printed(capfd, "fp8_fp4_gemm_nt")
    assert (int(cfg["BN"]), int(cfg["split"])) == (bn, split), cfg


def test_fp4_grouped_choices(fg, capfd, monkeypatch):
    monkeypatch.setenv("FG_PRINT_CONFIGS", "1")
    g, m_total, n, k = 32, 8192, 4096, 4096
    m_indices = (torch.arange(m_total, device="cuda", dtype=torch.int32) // 256).contiguous()
    d = torch.zeros((m_total, n), dtype=torch.bfloat16, device="cuda")
    fg.m_grouped_fp8_fp4_gemm_nt_contiguous(_u8(m_total, k), _i32(_cdiv(k, 512), _a4(m_total)), _u8(g, n, k // 2),
                                            _i32(g, k // 128, _a4(n)), m_indices, d)
    assert int(_printed(capfd, "m_grouped_fp8_fp4_nt_contiguous")["BN"]) == 224
    m_max, k2 = 256, 2048
    masked_m = torch.full((g,), 128, dtype=torch.int32, device="cuda")
    d2 = torch.zeros((g, m_max, n), dtype=torch.bfloat16, device="cuda")
    fg.m_grouped_fp8_fp4_gemm_nt_masked(_u8(g, m_max, k2), _i32(g, _cdiv(k2, 512), _a4(m_max)), _u8(g, n, k2 // 2),
                                        _i32(g, k2 // 128, _a4(n)), masked_m, d2, expected_m=128)
    assert int(_printed(capfd, "m_grouped_fp8_fp4_masked")["BN"]) == 224

