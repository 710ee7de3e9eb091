"""Test cases for the GPU parity tests: seeded draws from ``workloads`` encoded by the
oracle's quantiser, the oracle's expected values, and the comparison rule.

Tolerance (the stated accuracy target of the FP8 GEMM): per element
|d - ref| <= 1e-2 * |ref| + 1e-2 * rms(ref), and the normalised difference
1 - 2<x,y> / (|x|^2 + |y|^2) <= 1e-5, both over the valid rows only."""
from __future__ import annotations

import numpy as np

import oracle
import workloads
from oracle import formats as F
from oracle import fp4 as FP4

REL_TOL = 1e-2
DIFF_TOL = 1e-5
SENTINEL_BF16 = 0x7FBF
SENTINEL_F32 = 0x7FBFFFFF


def compare(got: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return {"n": 0}
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = np.abs(got - ref)
    bound = REL_TOL * np.abs(ref) + REL_TOL * rms
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), (f"{what}: element {worst} got {got[worst]} ref {ref[worst]} "
                                  f"(bound {bound[worst]:.3g}); {int((err > bound).sum())} bad of {ref.size}")
    denom = float(np.dot(got, got) + np.dot(ref, ref))
    diff = 0.0 if denom == 0 else 1.0 - 2.0 * float(np.dot(got, ref)) / denom
    assert diff <= DIFF_TOL, f"{what}: normalised difference {diff:.3g} > {DIFF_TOL}"
    return {"n": ref.size, "max_rel_to_rms": float(err.max() / max(rms, 1e-300)), "diff": diff}


# ------------------------------------------------------------------ dense
def dense_case(seed, m, n, k, with_c, out="bf16"):
    w = workloads.dense(seed, m, n, k, with_c)
    a, sa = F.quantize_rows(w["a"])
    b, sb = F.quantize_blocks(w["b"])
    return {"m": m, "n": n, "k": k, "a": a, "sfa": F.pack_ue8m0(sa), "b": b, "sfb": F.pack_ue8m0(sb),
            "c": w["c"], "out": out}


def dense_ref(case, rows=None):
    return oracle.fp8_gemm_nt(case["a"], case["sfa"], case["b"], case["sfb"], case["c"], rows=rows)


# ------------------------------------------------------------- contiguous
def contiguous_case(seed, weights="fp8", **kw):
    """weights: "fp8" (E4M3, 128x128-block scales) or "fp4" (packed E2M1, 1x32 scales)."""
    w = workloads.contiguous(seed, **kw)
    m_indices = w["m_indices"]
    m_total = len(m_indices)
    k = w["x"].shape[1]
    valid = w["row_token"] >= 0
    a = w["garbage"].copy()
    sa = w["garbage_sf"].copy()
    qa, qsa = F.quantize_rows(w["x"][w["row_token"][valid]])
    a[valid] = qa
    sa[valid] = qsa
    g_count, n, _ = w["b"].shape
    if weights == "fp4":
        bq, sfb = _mxfp4_experts(w["b"])
    else:
        bq = np.empty((g_count, n, k), np.uint8)
        sfb = []
        for e in range(g_count):
            bq[e], sb = F.quantize_blocks(w["b"][e])
            sfb.append(F.pack_ue8m0(sb))
        sfb = np.stack(sfb)
    return {"m_total": m_total, "n": n, "k": k, "g": g_count, "a": a, "sfa": F.pack_ue8m0(sa),
            "b": bq, "sfb": sfb, "m_indices": m_indices, "counts": w["counts"]}


def contiguous_ref(case, rows=None):
    return oracle.m_grouped_fp8_gemm_nt_contiguous(case["a"], case["sfa"], case["b"], case["sfb"],
                                                   case["m_indices"], rows=rows)


# ----------------------------------------------------------------- masked
def masked_case(seed, weights="fp8", **kw):
    """weights: "fp8" (E4M3, 128x128-block scales) or "fp4" (packed E2M1, 1x32 scales)."""
    w = workloads.masked(seed, **kw)
    g_count, m_max, k = w["x"].shape
    n = w["b"].shape[1]
    a = w["garbage"].copy()
    sfa = []
    bq = np.empty((g_count, n, k), np.uint8)
    sfb = []
    for e in range(g_count):
        mm = int(w["masked_m"][e])
        sa = w["garbage_sf"][e].copy()
        if mm > 0:
            qa, qsa = F.quantize_rows(w["x"][e, :mm])
            a[e, :mm] = qa
            sa[:mm] = qsa
        sfa.append(F.pack_ue8m0(sa))
        if weights != "fp4":
            bq[e], sb = F.quantize_blocks(w["b"][e])
            sfb.append(F.pack_ue8m0(sb))
    if weights == "fp4":
        bq, sfb = _mxfp4_experts(w["b"])
    else:
        sfb = np.stack(sfb)
    return {"g": g_count, "m_max": m_max, "n": n, "k": k, "a": a, "sfa": np.stack(sfa), "b": bq,
            "sfb": sfb, "masked_m": w["masked_m"]}


def masked_ref(case, experts=None, rows=None):
    return oracle.m_grouped_fp8_gemm_nt_masked(case["a"], case["sfa"], case["b"], case["sfb"],
                                               case["masked_m"], experts=experts, rows=rows)


# -------------------------------------------------------------- K-grouped
def k_grouped_case(seed, with_c=True, **kw):
    w = workloads.k_grouped(seed, **kw)
    a, sa = F.quantize_cols(w["a"])
    b, sb = F.quantize_cols(w["b"])
    return {"g": len(w["ks"]), "m": w["a"].shape[1], "n": w["b"].shape[1], "k_total": w["a"].shape[0],
            "a": a, "sfa": F.pack_ue8m0(sa), "b": b, "sfb": F.pack_ue8m0(sb), "ks": w["ks"],
            "c": w["c"] if with_c else None}


def k_grouped_ref(case, experts=None, rows=None):
    return oracle.k_grouped_fp8_gemm_tn_contiguous(case["a"], case["sfa"], case["b"], case["sfb"],
                                                   case["ks"], case["c"], experts=experts, rows=rows)


# -------------------------------------------------------------- FP8 x FP4
def _mxfp4_experts(b):
    """Weights [G, N, K] -> packed E2M1 [G, N, K/2] and packed 1x32 scale words per expert."""
    packed, words = [], []
    for e in range(b.shape[0]):
        q, sf = FP4.quantize_mxfp4(b[e])
        packed.append(q)
        words.append(FP4.pack_mx_scales(sf))
    return np.stack(packed), np.stack(words)


def fp4_dense_case(seed, m, n, k, with_c, out="bf16"):
    w = workloads.dense(seed, m, n, k, with_c)
    a, sa = F.quantize_rows(w["a"])
    b, sb = FP4.quantize_mxfp4(w["b"])
    return {"m": m, "n": n, "k": k, "a": a, "sfa": F.pack_ue8m0(sa), "b": b, "sfb": FP4.pack_mx_scales(sb),
            "c": w["c"], "out": out}


def fp4_dense_ref(case, rows=None):
    return oracle.fp8_fp4_gemm_nt(case["a"], case["sfa"], case["b"], case["sfb"], case["c"], rows=rows)


def fp4_contiguous_case(seed, **kw):
    """The contiguous routing and activations of :func:`contiguous_case` with MXFP4 weights."""
    return contiguous_case(seed, weights="fp4", **kw)


def fp4_contiguous_ref(case, rows=None):
    return oracle.m_grouped_fp8_fp4_gemm_nt_contiguous(case["a"], case["sfa"], case["b"], case["sfb"],
                                                       case["m_indices"], rows=rows)


def fp4_masked_case(seed, **kw):
    """The masked activations of :func:`masked_case` with MXFP4 weights."""
    return masked_case(seed, weights="fp4", **kw)


def fp4_masked_ref(case, experts=None, rows=None):
    return oracle.m_grouped_fp8_fp4_gemm_nt_masked(case["a"], case["sfa"], case["b"], case["sfb"],
                                                   case["masked_m"], experts=experts, rows=rows)


def decode_out(arr: np.ndarray, out: str) -> np.ndarray:
    """GPU output (bf16 bits as uint16/int16, or float32) to float64."""
    if out == "bf16":
        return F.bf16_to_f64(arr.view(np.uint16))
    return arr.astype(np.float64)


# ----------------------------------------------------------- other layouts
def layout_case(seed, layout, m, n, k, with_c, out="bf16"):
    """A dense case with the operands stored in `layout` ("nn", "tn", "tt"): A as [K, M]
    for a leading "t", B as [K, N] for a trailing "n" (same values as the NT case)."""
    case = dense_case(seed, m, n, k, with_c, out)
    a_t, b_n = layout[0] == "t", layout[1] == "n"
    case["layout"] = layout
    case["a_stored"] = np.ascontiguousarray(case["a"].T) if a_t else case["a"]
    case["b_stored"] = np.ascontiguousarray(case["b"].T) if b_n else case["b"]
    return case


def layout_ref(case, rows=None):
    fn = {"nn": oracle.fp8_gemm_nn, "tn": oracle.fp8_gemm_tn, "tt": oracle.fp8_gemm_tt}[case["layout"]]
    return fn(case["a_stored"], case["sfa"], case["b_stored"], case["sfb"], case["c"], rows=rows)


# ------------------------------------------------------------- MQA logits
def mqa_case(seed, s_len, t_len, ranges="random", heads=64, dim=128):
    """Indexer inputs: q encoded to E4M3 as drawn (clipped to the E4M3 range); each key row
    x_t scaled by sf_t = amax_t / 448 (FP32) and encoded, so kv * sf restores x_t."""
    w = workloads.mqa(seed, s_len, t_len, heads, dim, ranges)
    q = F.f64_to_e4m3(np.clip(w["q"], -448, 448))
    sf = (np.abs(w["x"]).max(axis=1) / 448.0).astype(np.float32)
    kv = F.f64_to_e4m3(w["x"] / sf[:, None].astype(np.float64))
    return {"q": q, "kv": kv, "sf": sf, "w": w["w"], "ks": w["ks"], "ke": w["ke"]}


# ---------------------------------------------------- quantised SwiGLU output
def dequant_1x128(q, sf):
    """codes [R, I], scale bytes [R, I/128] -> float64 [R, I]"""
    return F.e4m3_to_f64(q) * np.repeat(F.ue8m0_to_f64(sf), 128, axis=1)


def compare_quantised(q, sf, q_ref, sf_ref, y_ref, what):
    """q, sf: kernel codes / scale bytes of the valid rows; *_ref: the oracle's; y_ref: the
    oracle's FP32-rounded SwiGLU values (before quantisation)."""
    assert q.shape == q_ref.shape and sf.shape == sf_ref.shape
    got, ref = dequant_1x128(q, sf), dequant_1x128(q_ref, sf_ref)
    scale = np.repeat(F.ue8m0_to_f64(np.maximum(sf, sf_ref)), 128, axis=1)
    rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    bound = 0.126 * np.abs(y_ref) + 2.0 ** -9 * scale + 1e-5 * rms
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs off by more than one E4M3 spacing"
    assert np.mean(q == q_ref) >= 0.99, f"{what}: only {np.mean(q == q_ref):.4f} of codes identical"
    assert np.mean(sf == sf_ref) >= 0.99, f"{what}: only {np.mean(sf == sf_ref):.4f} of scales identical"
