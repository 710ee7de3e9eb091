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


# ------------------------------------------------------------------ MXFP4
def _mxfp4_draw(seed, shape):
    """Normal draws over wide magnitude ranges per 32-block, with zero blocks, and values
    placed exactly on E2M1 rounding ties (between neighbours of the scaled grid)."""
    g = workloads.rng(seed)
    x = g.standard_normal(shape, dtype=np.float32)
    blocks = x.reshape(-1, 32)
    blocks *= (2.0 ** g.integers(-30, 30, (blocks.shape[0], 1))).astype(np.float32)
    blocks[::13] = 0.0
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    ties = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    for r in range(1, blocks.shape[0], 7):          # block max 6: scale 1, ties land exactly
        blocks[r, :7] = ties * np.where(r % 2, 1, -1)
        blocks[r, 7] = 6.0
        blocks[r, 8:] = np.clip(blocks[r, 8:], -6, 6)
    return x


@pytest.mark.parametrize("g,n,k", [(1, 1, 128), (2, 37, 384), (3, 200, 1024)])
def test_mxfp4_bit_exact(fg, g, n, k):
    from oracle import fp4 as FP4
    w = _mxfp4_draw(41 + n, (g, n, k))
    refs = [FP4.quantize_mxfp4(w[e]) for e in range(g)]
    words_ref = np.stack([FP4.pack_mx_scales(sf) for _, sf in refs])
    q = torch.empty((g, n, k // 2), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(words_ref.shape, dtype=torch.int32, device="cuda")
    fg.quantize_mxfp4(torch.from_numpy(w).cuda(), q, sf)
    assert np.array_equal(q.cpu().numpy(), np.stack([r[0] for r in refs]))
    assert np.array_equal(sf.cpu().numpy()[:, :, :n], words_ref[:, :, :n])


def test_mxfp4_weights_feed_the_fp8_fp4_gemm(fg):
    """Quantise A (1x128 E4M3) and B (MXFP4) with the library, run the FP8 x FP4 GEMM, and
    compare with the oracle GEMM on the oracle's own quantisation of the same draws."""
    import cases as C
    from oracle import fp4 as FP4
    m, n, k = 160, 320, 768
    case = C.fp4_dense_case(42, m, n, k, False, "bf16")
    w = workloads.dense(42, m, n, k, False)
    a = torch.from_numpy(w["a"].astype(np.float32)).cuda()
    b = torch.from_numpy(w["b"].astype(np.float32)).cuda()
    qa = torch.empty((m, k), dtype=torch.uint8, device="cuda")
    sfa = torch.zeros(case["sfa"].shape, dtype=torch.int32, device="cuda")
    qb = torch.empty((n, k // 2), dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(case["sfb"].shape, dtype=torch.int32, device="cuda")
    fg.quantize_1x128_rows(a, qa, sfa)
    fg.quantize_mxfp4(b, qb, sfb)
    assert np.array_equal(qb.cpu().numpy(), case["b"])
    d = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    fg.fp8_fp4_gemm_nt(qa, sfa, qb, sfb, d)
    st, detail = fg.get_device_error()
    assert st == 0, (st, hex(detail))
    C.compare(d.float().cpu().numpy(), C.fp4_dense_ref(case), "quantised FP8 x FP4")
    assert FP4.E2M1_MAX == 6.0
