"""The C-ABI library on a host without a GPU: it loads, exports every entry point that
include/fg.h declares, rejects bad arguments before touching the device, and fails
loudly (FG_ERR_CUDA) rather than computing anything when no device is present."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fg():
    import moe_fp8_e4m3_gb300 as lib
    return lib


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fg_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_four_gemms():
    names = declared_functions()
    for n in ["fg_fp8_gemm_nt", "fg_m_grouped_fp8_gemm_nt_contiguous",
              "fg_m_grouped_fp8_gemm_nt_masked", "fg_k_grouped_fp8_gemm_tn_contiguous"]:
        assert n in names


def test_library_exports_every_declared_symbol(fg):
    raw = ctypes.CDLL(fg.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(fg):
    assert set(declared_functions()) <= set(fg._SIGNATURES)


def test_pure_host_utilities(fg):
    assert fg.get_mk_alignment_for_contiguous_layout() == 128
    assert [fg.get_tma_aligned_size(x, 4) for x in (0, 1, 4, 5, 65)] == [0, 4, 4, 8, 68]
    assert fg.get_tma_aligned_size(3, 3) == -1
    assert fg.lib.fg_status_string(-5).decode().startswith("bounded wait")


def test_pdl_switch(fg):
    assert fg.get_pdl() is True            # enabled by default
    fg.set_pdl(False)
    assert fg.get_pdl() is False
    fg.set_pdl(True)
    assert fg.get_pdl() is True


FAKE = 1 << 20          # a 16-byte aligned non-null "device" address; never dereferenced


def _nt(fg, m=128, n=256, k=512, a=FAKE, sfa=FAKE, b=FAKE, sfb=FAKE, c=None, d=FAKE, dtype=0):
    return fg.lib.fg_fp8_gemm_nt(m, n, k, a, sfa, b, sfb, c, d, dtype, None)


@pytest.mark.parametrize("kw,want", [
    (dict(k=100), -1), (dict(k=0), -1), (dict(n=8), -1), (dict(n=20), -1), (dict(m=-1), -1),
    (dict(a=None), -1), (dict(d=None), -1), (dict(sfb=FAKE + 4), -1), (dict(a=FAKE + 8), -1),
    (dict(dtype=7), -1), (dict(c=FAKE, dtype=0), -2), (dict(c=FAKE + 4, dtype=1), -1),
])
def test_dense_argument_errors(fg, kw, want):
    assert _nt(fg, **kw) == want


def test_empty_problem_is_a_no_op(fg):
    assert _nt(fg, m=0) == 0


def test_grouped_argument_errors(fg):
    L = fg.lib
    # contiguous: M_total not a multiple of 128, G < 1, misaligned indices
    assert L.fg_m_grouped_fp8_gemm_nt_contiguous(100, 256, 128, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == -1
    assert L.fg_m_grouped_fp8_gemm_nt_contiguous(128, 256, 128, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == -1
    assert L.fg_m_grouped_fp8_gemm_nt_contiguous(128, 256, 128, 2, FAKE, FAKE, FAKE, FAKE, FAKE + 2, FAKE, 0, None) == -1
    assert L.fg_m_grouped_fp8_gemm_nt_contiguous(0, 256, 128, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == 0
    # masked: G out of range, null mask
    assert L.fg_m_grouped_fp8_gemm_nt_masked(0, 64, 256, 128, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, None) == -1
    assert L.fg_m_grouped_fp8_gemm_nt_masked(2000, 64, 256, 128, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, None) == -1
    assert L.fg_m_grouped_fp8_gemm_nt_masked(2, 64, 256, 128, FAKE, FAKE, FAKE, FAKE, None, 0, FAKE, 0, None) == -1
    # K-grouped: M not a multiple of 16, K_total not a multiple of 128, null ks
    assert L.fg_k_grouped_fp8_gemm_tn_contiguous(2, 100, 256, 256, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None) == -1
    assert L.fg_k_grouped_fp8_gemm_tn_contiguous(2, 128, 256, 200, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None) == -1
    assert L.fg_k_grouped_fp8_gemm_tn_contiguous(2, 128, 256, 256, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None) == -1


def test_fp4_argument_errors(fg):
    L = fg.lib
    # packed FP4 B must start on a 32-byte boundary (16 is not enough); the FP8 rules hold too
    assert L.fg_fp8_fp4_gemm_nt(128, 256, 512, FAKE, FAKE, FAKE + 16, FAKE, None, FAKE, 0, None) == -1
    assert L.fg_fp8_fp4_gemm_nt(128, 256, 200, FAKE, FAKE, FAKE, FAKE, None, FAKE, 0, None) == -1
    assert L.fg_fp8_fp4_gemm_nt(128, 256, 512, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == -2
    assert L.fg_fp8_fp4_gemm_nt(0, 256, 512, FAKE, FAKE, FAKE, FAKE, None, FAKE, 0, None) == 0
    assert L.fg_m_grouped_fp8_fp4_gemm_nt_contiguous(128, 256, 128, 2, FAKE, FAKE, FAKE + 16, FAKE, FAKE, FAKE, 0,
                                                     None) == -1
    assert L.fg_m_grouped_fp8_fp4_gemm_nt_contiguous(100, 256, 128, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0,
                                                     None) == -1
    assert L.fg_m_grouped_fp8_fp4_gemm_nt_masked(2, 64, 256, 128, FAKE, FAKE, FAKE + 16, FAKE, FAKE, 0, FAKE, 0,
                                                 None) == -1
    assert L.fg_m_grouped_fp8_fp4_gemm_nt_masked(2, 64, 256, 128, FAKE, FAKE, FAKE, FAKE, None, 0, FAKE, 0, None) == -1


def test_no_device_fails_loudly(fg):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid arguments: the library must report the missing device, not compute anything
    assert _nt(fg) == fg.FG_ERR_CUDA
    assert fg.lib.fg_get_num_sms() == -1
