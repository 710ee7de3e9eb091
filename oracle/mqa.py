"""MQA logits of the lightning indexer (fp8_mqa_logits), as a plain FP64 definition.

TEST INFRASTRUCTURE (oracle): see the header of ``oracle/formats.py`` for who may
import it.  Shares no code with the CUDA library.

What is computed ("DeepGEMM Documentation", section 11 "Use V3.2 MQA Kernels for
Indexers"; yuguo-Jack/DeepGEMM README, the non-paged MQA logits): inputs q, E4M3
[S, H, D]; kv, E4M3 [T, D] with one FP32 scale per kv token; weights, FP32 [S, H]; and
per query token i a kv range [ks[i], ke[i]).  For every j in that range

    out[i, j] = sum_h  relu( q[i, h, :] . (kv[j, :] * sf[j]) ) * weights[i, h]

and, with clean_logits, every other entry of out [S, T] is -inf (without it they are
left as they were).  Evaluated in FP64 from the exactly decoded E4M3 values.
"""
from __future__ import annotations

import numpy as np

from . import formats as F


def fp8_mqa_logits(q, kv, kv_sf, weights, ks, ke, clean_logits=True, rows=None):
    """q uint8 [S, H, D]; kv uint8 [T, D]; kv_sf float32 [T]; weights float32 [S, H];
    ks, ke int [S].  Returns float64 [len(rows), T]; entries outside [ks[i], ke[i]) are
    -inf with clean_logits, else NaN (meaning: not written)."""
    s_len, heads, dim = q.shape
    t_len = kv.shape[0]
    rows = np.arange(s_len) if rows is None else np.asarray(rows)
    kvd = F.e4m3_to_f64(kv) * np.asarray(kv_sf, np.float64)[:, None]          # [T, D]
    out = np.full((len(rows), t_len), -np.inf if clean_logits else np.nan)
    for r, i in enumerate(rows):
        lo, hi = max(int(ks[i]), 0), min(int(ke[i]), t_len)
        if hi <= lo:
            continue
        qd = F.e4m3_to_f64(q[i])                                                # [H, D]
        dots = qd @ kvd[lo:hi].T                                                # [H, hi - lo]
        out[r, lo:hi] = np.maximum(dots, 0.0).T @ np.asarray(weights[i], np.float64)
    return out
