"""CPU oracle for the fine-grained FP8 GEMM and its MoE variants.

TEST INFRASTRUCTURE.  This package is the slow, plain, FP64 statement of what the
CUDA library computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The CUDA
library never imports, links or calls it; the two share no code, and the only common
module is the seeded input generator ``workloads.py``, which holds none of the
method's arithmetic.

Every function here is pinned by ``tests/test_oracle_*.py`` (run with
``-m "not gpu"``) against library routines, closed forms, brute force on tiny inputs
and hand-derived fixtures under ``tests/golden/``.
"""
from . import formats, fp4, gemm, mqa, swiglu  # noqa: F401
from .formats import (e4m3_to_f64, f64_to_bf16, f64_to_e4m3, pack_ue8m0,  # noqa: F401
                      quantize_blocks, quantize_cols, quantize_rows, ue8m0_for_amax,
                      ue8m0_to_f64, unpack_ue8m0, bf16_to_f64, tma_aligned_size)
from .mqa import fp8_mqa_logits  # noqa: F401
from .gemm import (fp8_gemm_nn, fp8_gemm_nt, fp8_gemm_tn, fp8_gemm_tt,  # noqa: F401
                   k_grouped_fp8_gemm_tn_contiguous, m_grouped_fp8_gemm_nn_contiguous,
                   m_grouped_fp8_gemm_nt_contiguous, m_grouped_fp8_gemm_nt_masked, round_output)
from .fp4 import (fp8_fp4_gemm_nt, m_grouped_fp8_fp4_gemm_nt_contiguous,  # noqa: F401
                  m_grouped_fp8_fp4_gemm_nt_masked)
