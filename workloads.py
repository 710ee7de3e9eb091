"""Seeded synthetic workloads for the fine-grained FP8 GEMM and its MoE variants.

This module only draws random numbers and builds index structure (routing,
segment lengths, masks, padding garbage).  It holds none of the GEMM's arithmetic:
no FP8 or UE8M0 encoding, no scaling, no products.  The tests hand its draws to the
oracle's quantiser; the benchmark hands them to the library's own quantise kernels.

Every draw comes from ``numpy.random.Generator(PCG64(seed))`` so the same seed gives
the same data on x86 and on Arm.

Workloads (shapes and distributions of the five benchmark cases):

* dense:      A[M,K], B[N,K] ~ N(0,1); optional C[M,N] ~ N(0,1).
* contiguous: 8192 tokens x[T,K] ~ N(0,1); uniform logits over 256 experts, top-6;
              the rows routed to experts 0..G-1 are kept, grouped by expert in
              expert order, tokens ascending, each segment padded to a multiple of
              128 rows marked -1 (garbage bytes); B[G,N,K] ~ N(0, 0.02).
* masked:     G experts x M_max rows; valid rows x ~ N(0,1), masked_m[g] ~ U{0..M_max};
              rows at or beyond the mask hold random bytes (NaN codes included) and
              random scale bytes; B[G,N,K] ~ N(0, 0.02).
* k-grouped:  per-expert K lengths ~ Multinomial(K_sum, uniform), each padded up to a
              multiple of 128 with zero rows; A[K,M], B[K,N] ~ N(0,1); C[G,M,N] ~ N(0,1).
* mqa:        indexer queries q[S,H,D] ~ N(0, 16), keys x[T,D] ~ N(0,1), head weights
              w[S,H] ~ N(0,1); per-token kv ranges either causal (token i of S sees the
              last T-S+i+1 keys' prefix) or random, with a full, an empty and a
              clipped-past-T range planted in rows 0, 1, 2.
"""
from __future__ import annotations

import numpy as np

ALIGN = 128


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _normal(g: np.random.Generator, shape, std=1.0) -> np.ndarray:
    x = g.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def dense(seed: int, m: int, n: int, k: int, with_c: bool) -> dict:
    g = rng(seed)
    out = {"a": _normal(g, (m, k)), "b": _normal(g, (n, k)), "c": None}
    if with_c:
        out["c"] = _normal(g, (m, n))
    return out


def falling_sigmas(g: np.random.Generator, rows: int, groups: int, spread: int) -> np.ndarray:
    """Standard deviations 2^e for `rows` x `groups` blocks, e falling from +spread at the
    first 128-wide K-group to -spread at the last (linear trend), plus an integer jitter in
    [-2, 2] per block, clipped to [-spread, spread]."""
    trend = np.rint(spread * (1.0 - 2.0 * np.arange(groups) / max(groups - 1, 1)))
    e = np.clip(trend[None, :] + g.integers(-2, 3, (rows, groups)), -spread, spread)
    return np.exp2(e).astype(np.float32)


def dense_wide_range(seed: int, m: int, n: int, k: int, with_c: bool, spread: int = 10) -> dict:
    """Dense draws whose magnitude changes from one 128-wide K-group to the next: element
    (i, k) of A ~ N(0, s_a[i, k/128]^2) with s_a from ``falling_sigmas`` per row, element
    (j, k) of B ~ N(0, s_b[j/128, k/128]^2) per 128-row block; C ~ N(0, 1).  Products of
    the two span about 2 * spread binades either side of 1, largest in the first K-groups,
    so the smallest groups are accumulated last."""
    g = rng(seed)
    groups = k // ALIGN
    sa = np.repeat(falling_sigmas(g, m, groups, spread), ALIGN, axis=1)
    sb = np.repeat(np.repeat(falling_sigmas(g, (n + ALIGN - 1) // ALIGN, groups, spread), ALIGN, axis=0)[:n],
                   ALIGN, axis=1)
    out = {"a": _normal(g, (m, k)) * sa, "b": _normal(g, (n, k)) * sb, "c": None}
    if with_c:
        out["c"] = _normal(g, (m, n))
    return out


def k_grouped_wide_range(seed: int, ks, m: int, n: int, spread: int = 10) -> dict:
    """K-grouped draws (segments ``ks``, multiples of 128, no padding rows) with the
    magnitudes of ``dense_wide_range`` along the concatenated K axis: element (k, i) of A ~
    N(0, s_a[i, k/128]^2) per column i of A, likewise for B; C[G, M, N] ~ N(0, 1)."""
    g = rng(seed)
    ks = np.asarray(ks, dtype=np.int64)
    k_total = int(ks.sum())
    groups = k_total // ALIGN
    sa = np.repeat(falling_sigmas(g, m, groups, spread), ALIGN, axis=1).T
    sb = np.repeat(falling_sigmas(g, n, groups, spread), ALIGN, axis=1).T
    return {"a": _normal(g, (k_total, m)) * sa, "b": _normal(g, (k_total, n)) * sb,
            "ks": ks.astype(np.int32), "c": _normal(g, (len(ks), m, n))}


def routing(g: np.random.Generator, num_tokens: int, num_routed: int, topk: int, num_groups: int):
    """Uniform random logits, top-k experts per token; the rows routed to experts
    0..num_groups-1 grouped by expert (ascending token order), each segment padded to a
    multiple of 128 rows.  Returns (m_indices, row_token, counts)."""
    logits = g.random((num_tokens, num_routed), dtype=np.float32)
    top = np.argsort(-logits, axis=1, kind="stable")[:, :topk]
    m_indices, row_token, counts = [], [], []
    for e in range(num_groups):
        toks = np.nonzero((top == e).any(axis=1))[0]
        counts.append(len(toks))
        pad = (-len(toks)) % ALIGN
        m_indices += [e] * len(toks) + [-1] * pad
        row_token += list(toks) + [-1] * pad
    return (np.array(m_indices, dtype=np.int32), np.array(row_token, dtype=np.int64),
            np.array(counts, dtype=np.int64))


def contiguous(seed: int, num_tokens: int = 8192, num_routed: int = 256, topk: int = 6,
               num_groups: int = 32, n: int = 4096, k: int = 4096, b_std: float = 0.02) -> dict:
    """Routing structure and draws for the M-grouped contiguous layout.

    Returns x (token activations), ``row_token`` (token index of each valid row, or -1),
    ``m_indices`` (expert of each row, -1 for padding), per-expert ``counts``,
    ``garbage`` bytes and scale bytes for padding rows, and the expert weights ``b``."""
    g = rng(seed)
    x = _normal(g, (num_tokens, k))
    m_indices, row_token, counts = routing(g, num_tokens, num_routed, topk, num_groups)
    m_total = len(m_indices)
    return {
        "x": x,
        "m_indices": m_indices,
        "row_token": row_token,
        "counts": counts,
        "garbage": g.integers(0, 256, (m_total, k), dtype=np.uint8),
        "garbage_sf": g.integers(0, 256, (m_total, k // ALIGN), dtype=np.uint8),
        "b": _normal(g, (num_groups, n, k), b_std),
    }


def masked(seed: int, num_groups: int = 32, m_max: int = 256, n: int = 4096, k: int = 2048,
           b_std: float = 0.02, masked_m=None) -> dict:
    g = rng(seed)
    if masked_m is None:
        masked_m = g.integers(0, m_max + 1, num_groups)
    masked_m = np.asarray(masked_m, dtype=np.int32)
    return {
        "x": _normal(g, (num_groups, m_max, k)),
        "masked_m": masked_m,
        "garbage": g.integers(0, 256, (num_groups, m_max, k), dtype=np.uint8),
        "garbage_sf": g.integers(0, 256, (num_groups, m_max, k // ALIGN), dtype=np.uint8),
        "b": _normal(g, (num_groups, n, k), b_std),
    }


def k_grouped(seed: int, num_groups: int = 8, m: int = 4096, n: int = 2048,
              k_sum: int = 16384, ks=None) -> dict:
    """Per-expert K lengths and draws for the K-grouped weight-gradient GEMM.
    ``ks_true`` are the multinomial counts, ``ks`` the lengths padded to 128; the
    padding rows of A and B are zero."""
    g = rng(seed)
    if ks is None:
        ks_true = g.multinomial(k_sum, [1.0 / num_groups] * num_groups)
    else:
        ks_true = np.asarray(ks)
    ks_true = np.asarray(ks_true, dtype=np.int64)
    ks_pad = (ks_true + ALIGN - 1) // ALIGN * ALIGN
    k_total = int(ks_pad.sum())
    a = np.zeros((k_total, m), dtype=np.float32)
    b = np.zeros((k_total, n), dtype=np.float32)
    off = 0
    for e in range(num_groups):
        t = int(ks_true[e])
        a[off:off + t] = _normal(g, (t, m))
        b[off:off + t] = _normal(g, (t, n))
        off += int(ks_pad[e])
    return {"a": a, "b": b, "ks": ks_pad.astype(np.int32), "ks_true": ks_true,
            "c": _normal(g, (num_groups, m, n))}


def mqa(seed: int, s_len: int, t_len: int, heads: int = 64, dim: int = 128, ranges: str = "random") -> dict:
    g = rng(seed)
    q = g.standard_normal((s_len, heads, dim)) * 4.0
    x = g.standard_normal((t_len, dim))
    w = g.standard_normal((s_len, heads)).astype(np.float32)
    if ranges == "causal":
        ks = np.zeros(s_len, np.int32)
        ke = (np.arange(s_len) + 1 + (t_len - s_len)).astype(np.int32)
    else:
        lo = g.integers(-5, t_len + 5, s_len)
        hi = g.integers(-5, t_len + 40, s_len)
        ks, ke = np.minimum(lo, hi).astype(np.int32), np.maximum(lo, hi).astype(np.int32)
        ks[0], ke[0] = 0, t_len
        if s_len > 2:
            ks[1], ke[1] = 7, 7
            ks[2], ke[2] = t_len - 3, t_len + 100
    return {"q": q, "x": x, "w": w, "ks": ks, "ke": ke}


def device_normal(seed: int, shape, std: float = 1.0, device: str = "cuda"):
    """N(0, std^2) float32 draws made on the GPU by torch's seeded generator, for
    benchmark inputs too large to draw on the host.  (Seeded and reproducible on one
    machine; not the same numbers as the numpy draws above.)"""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def device_bytes(seed: int, shape, device: str = "cuda"):
    """Uniform random bytes on the GPU (garbage rows)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randint(0, 256, tuple(shape), generator=gen, device=device, dtype=torch.uint8)
