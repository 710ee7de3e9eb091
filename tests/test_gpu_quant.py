"""GPU quantise/pack kernels against the oracle's quantiser: bit-exact codes and packed
scale words (the decision of each code is taken in the same precision on both sides:
the oracle rounds the exact x / 2^e, the kernel rounds the exact FP32 x * 2^-e)."""
import numpy as np
import pytest

import workloads
from oracle import formats as F

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_fp8_e4m3_gb300 as lib
    return lib


def _draw(seed, shape, spread=True):
    g = workloads.rng(seed)
    x = g.standard_normal(shape, dtype=np.float32)
    if spread:   # groups of very different magnitudes, zeros and exact ties
        x *= (10.0 ** g.integers(-6, 6, shape[:-1] + (1,))).astype(np.float32)
        x.reshape(-1)[::97] = 0.0
    return x


def _zero_group(x):
    x[0, :128] = 0.0
    return x


@pytest.mark.parametrize("rows,k", [(1, 128), (37, 640), (256, 4096), (130, 384)])
def test_rows_bit_exact(fg, rows, k):
    x = _zero_group(_draw(1 + rows, (rows, k)))
    q_ref, sf_ref = F.quantize_rows(x)
    words_ref = F.pack_ue8m0(sf_ref)
    xt = torch.from_numpy(x).cuda()
    q = torch.empty((rows, k), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(words_ref.shape, dtype=torch.int32, device="cuda")
    fg.quantize_1x128_rows(xt, q, sf)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sf.cpu().numpy(), words_ref)


@pytest.mark.parametrize("g,n,k", [(1, 128, 128), (3, 200, 640), (2, 256, 1024)])
def test_blocks_bit_exact(fg, g, n, k):
    w = _draw(7 + n, (g, n, k))
    w[0, :128, :128] = 0.0
    refs = [F.quantize_blocks(w[e]) for e in range(g)]
    words_ref = np.stack([F.pack_ue8m0(sf) for _, sf in refs])
    q = torch.empty((g, n, k), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(words_ref.shape, dtype=torch.int32, device="cuda")
    fg.quantize_128x128_blocks(torch.from_numpy(w).cuda(), q, sf)
    assert np.array_equal(q.cpu().numpy(), np.stack([r[0] for r in refs]))
    assert np.array_equal(sf.cpu().numpy(), words_ref)


@pytest.mark.parametrize("k,mn", [(128, 16), (640, 208), (2048, 512)])
def test_cols_bit_exact(fg, k, mn):
    x = _draw(11 + k, (mn, k)).T.copy()          # groups along the leading axis
    x[:128, 0] = 0.0
    q_ref, sf_ref = F.quantize_cols(x)
    words_ref = F.pack_ue8m0(sf_ref)
    q = torch.empty((k, mn), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(words_ref.shape, dtype=torch.int32, device="cuda")
    fg.quantize_1x128_cols(torch.from_numpy(x).cuda(), q, sf)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sf.cpu().numpy(), words_ref)


def test_quantised_operands_feed_the_gemm(fg):
    """End to end on the device: quantise A and B with the library, run the GEMM, and
    compare with the oracle GEMM fed by the oracle's own quantisation of the same draws."""
    import cases as C
    m, n, k = 192, 256, 512
    case = C.dense_case(21, m, n, k, True, "f32")
    w = workloads.dense(21, m, n, k, True)
    a = torch.empty((m, k), dtype=torch.uint8, device="cuda")
    sfa = torch.zeros(case["sfa"].shape, dtype=torch.int32, device="cuda")
    b = torch.empty((n, k), dtype=torch.uint8, device="cuda")
    sfb = torch.zeros((1,) + case["sfb"].shape, dtype=torch.int32, device="cuda")
    fg.quantize_1x128_rows(torch.from_numpy(w["a"]).cuda(), a, sfa)
    fg.quantize_128x128_blocks(torch.from_numpy(w["b"]).cuda(), b, sfb)
    d = torch.empty((m, n), dtype=torch.float32, device="cuda")
    fg.fp8_gemm_nt(a, sfa, b, sfb[0], d, c=torch.from_numpy(w["c"]).cuda())
    C.compare(d.cpu().numpy(), C.dense_ref(case), "quantise + GEMM")
