"""GPU parity of the lightning-indexer MQA logits (fp8_mqa_logits) against the oracle.

In-range logits are compared with the GEMM tolerance (FP32 accumulation against the FP64
definition); entries outside [ks[i], ke[i]) must be exactly -inf with clean_logits and
bit-for-bit untouched without it."""
import numpy as np
import pytest

import cases as C
from oracle import mqa as MQ

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

H, D = 64, 128
SENT = 0x7FBFFFFF          # NaN pattern


@pytest.fixture(scope="module")
def fg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_fp8_e4m3_gb300 as lib
    return lib


def _ok(fg):
    st, detail = fg.get_device_error()
    assert st == 0, (st, hex(detail))


mqa_case = C.mqa_case


def run(fg, case, clean=True):
    from gpu_util import dev
    s_len, t_len = case["q"].shape[0], case["kv"].shape[0]
    out = torch.full((s_len, t_len), SENT, dtype=torch.int32, device="cuda").view(torch.float32)
    fg.fp8_mqa_logits(dev(case["q"]), dev(case["kv"]), dev(case["sf"]), dev(case["w"]), dev(case["ks"]),
                      dev(case["ke"]), out, clean_logits=clean)
    _ok(fg)
    return out.cpu().numpy()


def check(case, got, clean, rows=None):
    ref = MQ.fp8_mqa_logits(case["q"], case["kv"], case["sf"], case["w"], case["ks"], case["ke"], clean, rows=rows)
    got = got if rows is None else got[rows]
    inside = np.isfinite(ref)
    C.compare(got[inside], ref[inside], "mqa logits in range")
    if clean:
        assert np.all(np.isneginf(got[~inside])), "out-of-range logits not -inf"
    else:
        bits = got.view(np.uint32)
        assert np.all(bits[~inside] == SENT), "out-of-range logits written"


@pytest.mark.parametrize("s_len,t_len", [(37, 300), (2, 128), (64, 1000)])
@pytest.mark.parametrize("clean", [True, False])
def test_mqa_logits_random_ranges(fg, s_len, t_len, clean):
    case = mqa_case(100 + s_len + t_len, s_len, t_len)
    check(case, run(fg, case, clean), clean)


def test_mqa_logits_causal(fg):
    case = mqa_case(7, 512, 640, "causal")
    check(case, run(fg, case, True), True)


def test_mqa_logits_nonpositive_scales(fg):
    """kv scales of either sign and zero: relu applies to the scaled dot product."""
    case = mqa_case(11, 20, 256)
    case["sf"] = case["sf"] * np.where(np.arange(256) % 3 == 0, -1.0, 1.0).astype(np.float32)
    case["sf"][5] = 0.0
    check(case, run(fg, case, True), True)


def test_mqa_logits_closed_form(fg):
    """All-ones q and kv: out[i, j] = D * sf[j] * sum_h w[i, h] exactly (products and sums
    of small integers and powers of two are exact in FP32)."""
    s_len, t_len = 9, 200
    g = np.random.Generator(np.random.PCG64(3))
    case = {"q": np.full((s_len, H, D), 0x38, np.uint8), "kv": np.full((t_len, D), 0x38, np.uint8),
            "sf": (2.0 ** g.integers(-4, 4, t_len)).astype(np.float32),
            "w": g.integers(-8, 9, (s_len, H)).astype(np.float32),
            "ks": np.zeros(s_len, np.int32), "ke": np.full(s_len, t_len, np.int32)}
    got = run(fg, case, True)
    want = D * case["sf"][None, :].astype(np.float64) * case["w"].sum(axis=1, dtype=np.float64)[:, None]
    assert np.array_equal(got.astype(np.float64), want)


def test_mqa_logits_unsupported_shape(fg):
    assert fg.lib.fg_fp8_mqa_logits(4, 8, 32, 128, 16, 16, 16, 16, 16, 16, 1, 16, None) == fg.FG_ERR_UNSUPPORTED
