#!/usr/bin/env python
"""Benchmark of the fine-grained FP8 GEMM library on one GB300 (or N replicas).

Default workload (the headline metric's configuration): the dense FP8 NT GEMM pair
  prefill  M=4096 N=7168 K=2048
  decode   M=64   N=7168 K=4096
with A scaled per 1x128 row group, B per 128x128 block (UE8M0), and an FP32 C
accumulated into an FP32 D.  One step = one call of each.  Inputs are N(0,1) draws
from a seeded torch generator on the GPU, quantised by the library's own quantise
kernels.  L2 rule (--l2 auto): a workload whose step moves more than twice the L2 size
(the dense pair: 291 MB against 129 MB; the grouped configurations too) runs back to back
without a flush, since nothing of one step survives in L2 to the next; a smaller one (the
128x256x512 case) has L2 flushed before every timed step (a write of twice its size),
outside the timed events.  --l2 flush forces the flush everywhere.

Two kinds of timed passes of --steps steps each, each repeated back to back until the
timed region lasts at least MIN_TIMED_SECONDS (so that the clock sampler sees it):
  1. the step time (the headline value): CUDA events only at the step boundaries, so the
     GEMMs of a step run back to back as a caller issues them (programmatic dependent
     launch lets the second start while the first drains);
  2. the per-kernel durations (the roofline and the per-kernel breakdown): an event
     between consecutive GEMMs, which serialises them.
The default run then times the other benchmark configurations on the same rules (one
pass each) and records them in config.kernels: the small dense case (configuration 0,
launch latency), the M-grouped contiguous (2), masked (3) and K-grouped (4) GEMMs.  Each
kernel entry gives its fraction of the stated roofs (8 TB/s HBM, 4.5 PFLOP/s dense FP8)
and of the measured ones (MEASURED_PEAKS.json copy bandwidth; BF16 burst x 2 for FP8).

Other workloads (--workload prefill | decode | small | contiguous | masked | k_grouped,
the other operand layouts prefill_nn | prefill_tn | prefill_tt | contiguous_nn, the fused
gate-up GEMM contiguous_swiglu, the indexer's mqa_logits, the quantisers quant, the FP8 x
FP4 forms fp4_dense_pair | fp4_prefill | fp4_decode | fp4_contiguous | fp4_masked |
fp4_contiguous_swiglu, and the MoE expert MLP moe_mlp | fp4_moe_mlp) time them on the same
rules; they are measurement aids, the default line is the headline (its config.kernels also
records small, contiguous, masked, k_grouped, quant and the FP8 x FP4 dense pair,
contiguous and masked).

Output: one JSON line from rank 0 (see the keys below).  ``--impl reference`` times the
CPU oracle instead, on full dense-pair steps (or a bounded sample of each step when
that many full steps would not end within a few minutes).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 GEMM TFLOPS (and HBM GB/s for small M) at 1 GB300 vs roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0          # nominal dense ratio (4.5 / 2.25 PFLOP/s)
KERNEL_SOURCES = ["fg_gemm_kernel.cuh", "fg_ptx.cuh", "fg_gemm_inst.cuh", "fg_gemm_nt.cu", "fg_gemm_split.cu",
                  "fg_gemm_tn.cu", "fg_gemm_layouts.cu", "fg_gemm_sepc.cu", "fg_gemm_dense.cu", "fg_gemm_swiglu.cu", "fg_fp8.cuh", "fg_mqa.cu",
                  "fg_gemm_fp4.cu", "fg_gemm_fp4_grouped.cu"]


def align4(x: int) -> int:
    return (x + 3) // 4 * 4


def cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


# --------------------------------------------------------------------------- peaks
def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:  # noqa: BLE001
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "moe_fp8_e4m3_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))[workload][kernel]
    except Exception:  # noqa: BLE001
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clock sampling
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:  # noqa: BLE001
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [r for (t, r) in self.rows if t0 - 0.05 <= t <= t1 + 0.05]
        note = "samples inside the timed region"
        if not inside:
            inside = [r for (_, r) in self.rows]
            note = "timed region shorter than the sampling interval: samples around it"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = sorted(v for v in (num(r[2]) for r in inside) if v is not None)
        mx = [num(r[3]) for r in inside if num(r[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for i, nm in enumerate(names):
                if r[6 + i].lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside), "note": note,
                "power_w_max": max((num(r[4]) or 0.0) for r in inside)}


# ---------------------------------------------------------------------- workloads
class DensePair:
    """The headline workload: dense NT prefill + decode GEMMs, FP32 C -> FP32 D."""
    name = "dense_pair"
    description = ("dense FP8 NT GEMM pair: prefill M=4096 N=7168 K=2048 + decode M=64 N=7168 K=4096; "
                   "A 1x128 / B 128x128 UE8M0 scales; FP32 C accumulated into FP32 D")
    SHAPES = [("prefill", 4096, 7168, 2048), ("decode", 64, 7168, 4096)]
    WITH_C = True        # FP32 C accumulated into an FP32 D (else no C and a BF16 D)
    PREFIX = ""          # kernel-name prefix in the per-kernel table

    @staticmethod
    def make_weights(torch, fg, xb, n, k):
        """E4M3 weights with one scale per 128x128 block (the library's quantiser)."""
        b = torch.empty((n, k), dtype=torch.uint8, device="cuda")
        sfb = torch.zeros((1, cdiv(k, 512), align4(cdiv(n, 128))), dtype=torch.int32, device="cuda")
        fg.quantize_128x128_blocks(xb, b, sfb)
        return b, sfb[0]

    def __init__(self, torch, fg, seed):
        import workloads
        self.torch, self.fg = torch, fg
        self.parts = []
        for i, (nm, m, n, k) in enumerate(self.SHAPES):
            xa = workloads.device_normal(seed + 10 * i, (m, k))
            xb = workloads.device_normal(seed + 10 * i + 1, (n, k))
            c = workloads.device_normal(seed + 10 * i + 2, (m, n)) if self.WITH_C else None
            a = torch.empty((m, k), dtype=torch.uint8, device="cuda")
            sfa = torch.zeros((cdiv(k, 512), align4(m)), dtype=torch.int32, device="cuda")
            fg.quantize_1x128_rows(xa, a, sfa)
            b, sfb = self.make_weights(torch, fg, xb, n, k)
            del xa, xb
            d = torch.empty((m, n), dtype=torch.float32 if self.WITH_C else torch.bfloat16, device="cuda")
            flops = 2.0 * m * n * k
            nbytes = (m * k + b.numel() + sfa.numel() * 4 + sfb.numel() * 4 + (m * n * 4 if self.WITH_C else 0)
                      + m * n * d.element_size())
            self.parts.append({"name": self.PREFIX + nm, "m": m, "n": n, "k": k, "a": a, "sfa": sfa, "b": b,
                               "sfb": sfb, "c": c, "d": d, "flops": flops, "bytes": nbytes})
        torch.cuda.synchronize()

    def launches(self):
        return [lambda p=p: self.fg.fp8_gemm_nt(p["a"], p["sfa"], p["b"], p["sfb"], p["d"], c=p["c"])
                for p in self.parts]

    def e2e_io(self):
        """(inputs as (device tensor, pinned host copy)), (outputs likewise)."""
        ins, outs = [], []
        for p in self.parts:
            for key in ("a", "sfa", "b", "sfb", "c"):
                if p[key] is not None:
                    ins.append((p[key], p[key].cpu().pin_memory()))
            outs.append((p["d"], self.torch.empty_like(p["d"], device="cpu").pin_memory()))
        return ins, outs

    def e2e_double(self):
        """Two device sets of every operand and output, for the double-buffered end-to-end
        loop: returns (bind(k), [(inputs, outputs) of set 0, of set 1]).  bind(k) points the
        launches at set k; both sets copy from and to the same pinned host buffers."""
        keys_in = ("a", "sfa", "b", "sfb", "c")
        sets = [{}, {}]
        io = [([], []), ([], [])]
        for j, p in enumerate(self.parts):
            host_in = {key: p[key].cpu().pin_memory() for key in keys_in if p[key] is not None}
            host_out = self.torch.empty_like(p["d"], device="cpu").pin_memory()
            for k in (0, 1):
                dev = {key: (p[key] if k == 0 else (p[key].clone() if p[key] is not None else None))
                       for key in keys_in + ("d",)}
                sets[k][j] = dev
                io[k][0].extend((dev[key], host_in[key]) for key in keys_in if dev[key] is not None)
                io[k][1].append((dev["d"], host_out))

        def bind(k):
            for j, p in enumerate(self.parts):
                p.update(sets[k][j])
        return bind, io

    _oracle_inputs = None

    @classmethod
    def oracle_inputs(cls):
        """The same shapes for the CPU oracle: seeded numpy draws quantised by the oracle
        (made once per process)."""
        if cls._oracle_inputs is not None:
            return cls._oracle_inputs
        from oracle import formats as F
        import workloads
        out = []
        for i, (nm, m, n, k) in enumerate(cls.SHAPES):
            w = workloads.dense(2000 + i, m, n, k, True)
            a, sa = F.quantize_rows(w["a"])
            b, sb = F.quantize_blocks(w["b"])
            out.append({"m": m, "n": n, "k": k, "a": a, "sa": sa, "b": b, "sb": sb, "c": w["c"]})
        cls._oracle_inputs = out
        return out

    @classmethod
    def oracle_full_step(cls):
        """One full step of the oracle (both GEMMs, every output)."""
        import oracle
        from oracle import formats as F
        items = []
        for t in cls.oracle_inputs():
            sfa, sfb = F.pack_ue8m0(t["sa"]), F.pack_ue8m0(t["sb"])
            items.append((lambda t=t, sfa=sfa, sfb=sfb: oracle.fp8_gemm_nt(t["a"], sfa, t["b"], sfb, t["c"]),
                          2.0 * t["m"] * t["n"] * t["k"]))
        return items, "one full step (prefill 4096x7168x2048 + decode 64x7168x4096) per repetition"

    @classmethod
    def oracle_sub_step(cls, rows=32, cols=256):
        """A bounded sample of one step: the first `rows` x `cols` outputs of each GEMM,
        computed by the oracle on the corresponding slices of A, B, C and their scales."""
        import oracle
        from oracle import formats as F
        items = []
        for t in cls.oracle_inputs():
            r, c = min(rows, t["m"]), min(cols, t["n"])
            a, sfa = t["a"][:r], F.pack_ue8m0(t["sa"][:r])
            b, sfb = t["b"][:c], F.pack_ue8m0(t["sb"][:cdiv(c, 128)])
            cc = t["c"][:r, :c].copy()
            items.append((lambda a=a, sfa=sfa, b=b, sfb=sfb, cc=cc: oracle.fp8_gemm_nt(a, sfa, b, sfb, cc),
                          2.0 * r * c * t["k"]))
        return items, f"per step: the first {rows} rows x {cols} columns of the prefill and decode outputs"


class Contiguous:
    name = "contiguous"
    description = ("M-grouped contiguous FP8 NT GEMM: 32 experts of 256 (top-6 of 8192 tokens, experts 0-31 "
                   "kept, 128-row padded segments, -1 padding rows), N=4096 K=4096, BF16 D")

    def __init__(self, torch, fg, seed):
        import numpy as np
        import workloads
        self.torch, self.fg = torch, fg
        m_indices, row_token, counts = workloads.routing(workloads.rng(seed), 8192, 256, 6, 32)
        m_total, n, k, g = len(m_indices), 4096, 4096, 32
        x = workloads.device_normal(seed + 1, (8192, k))
        xa = torch.zeros((m_total, k), dtype=torch.float32, device="cuda")
        valid = np.nonzero(row_token >= 0)[0]
        xa[torch.from_numpy(valid).cuda()] = x[torch.from_numpy(row_token[valid]).cuda()]
        del x
        self.a = torch.empty((m_total, k), dtype=torch.uint8, device="cuda")
        self.sfa = torch.zeros((cdiv(k, 512), align4(m_total)), dtype=torch.int32, device="cuda")
        fg.quantize_1x128_rows(xa, self.a, self.sfa)
        del xa
        pad = torch.from_numpy(np.nonzero(row_token < 0)[0]).cuda()
        self.a[pad] = workloads.device_bytes(seed + 2, (len(pad), k))
        self.b, self.sfb = self.make_expert_weights(torch, fg, seed, g, n, k)
        self.m_indices = torch.from_numpy(m_indices).cuda()
        self.d = torch.empty((m_total, n), dtype=torch.bfloat16, device="cuda")
        nv = int(counts.sum())
        used = int((counts > 0).sum())
        self.nv, self.used = nv, used
        self.flops = 2.0 * nv * n * k
        self.bytes = (nv * k + used * self.b[0].numel() + self.sfb.numel() * 4 + self.sfa.numel() * 4 + nv * n * 2
                      + m_total * 4)
        self.parts = [{"name": self.name, "flops": self.flops, "bytes": self.bytes}]
        torch.cuda.synchronize()

    @staticmethod
    def make_expert_weights(torch, fg, seed, g, n, k):
        """Per expert: N(0, 0.02^2) draws, E4M3 with one scale per 128x128 block."""
        import workloads
        b = torch.empty((g, n, k), dtype=torch.uint8, device="cuda")
        sfb = torch.zeros((g, cdiv(k, 512), align4(cdiv(n, 128))), dtype=torch.int32, device="cuda")
        for e in range(g):
            xb = workloads.device_normal(seed + 100 + e, (1, n, k), std=0.02)
            fg.quantize_128x128_blocks(xb, b[e:e + 1], sfb[e:e + 1])
        return b, sfb

    def launches(self):
        return [lambda: self.fg.m_grouped_fp8_gemm_nt_contiguous(self.a, self.sfa, self.b, self.sfb,
                                                                 self.m_indices, self.d)]

    def e2e_io(self):
        ins = [(t, t.cpu().pin_memory()) for t in (self.a, self.sfa, self.b, self.sfb, self.m_indices)]
        return ins, [(self.d, self.torch.empty_like(self.d, device="cpu").pin_memory())]



class Masked:
    name = "masked"
    description = ("M-grouped masked FP8 NT GEMM: 32 experts x 256 rows, masked_m ~ U{0..256} on the device, "
                   "N=4096 K=2048, BF16 D")
    make_expert_weights = staticmethod(Contiguous.make_expert_weights)

    def __init__(self, torch, fg, seed):
        import numpy as np
        import workloads
        self.torch, self.fg = torch, fg
        g, m_max, n, k = 32, 256, 4096, 2048
        mm = workloads.rng(seed).integers(0, m_max + 1, g).astype(np.int32)
        x = workloads.device_normal(seed + 1, (g * m_max, k))
        self.a = torch.empty((g, m_max, k), dtype=torch.uint8, device="cuda")
        self.sfa = torch.zeros((g, cdiv(k, 512), align4(m_max)), dtype=torch.int32, device="cuda")
        for e in range(g):
            fg.quantize_1x128_rows(x[e * m_max:(e + 1) * m_max], self.a[e], self.sfa[e])
            if mm[e] < m_max:
                self.a[e, mm[e]:] = workloads.device_bytes(seed + 50 + e, (m_max - mm[e], k))
        del x
        self.b, self.sfb = self.make_expert_weights(torch, fg, seed, g, n, k)
        self.masked_m = torch.from_numpy(mm).cuda()
        self.d = torch.empty((g, m_max, n), dtype=torch.bfloat16, device="cuda")
        nv = int(mm.sum())
        used = int((mm > 0).sum())
        self.flops = 2.0 * nv * n * k
        self.bytes = nv * k + used * self.b[0].numel() + nv * n * 2 + self.sfa.numel() * 4 + self.sfb.numel() * 4
        self.parts = [{"name": self.name, "flops": self.flops, "bytes": self.bytes}]
        self.expected_m = int(mm.mean())
        torch.cuda.synchronize()

    def launches(self):
        return [lambda: self.fg.m_grouped_fp8_gemm_nt_masked(self.a, self.sfa, self.b, self.sfb, self.masked_m,
                                                             self.d, expected_m=self.expected_m)]

    def e2e_io(self):
        ins = [(t, t.cpu().pin_memory()) for t in (self.a, self.sfa, self.b, self.sfb, self.masked_m)]
        return ins, [(self.d, self.torch.empty_like(self.d, device="cpu").pin_memory())]


class KGrouped:
    name = "k_grouped"
    description = ("K-grouped contiguous FP8 TN GEMM: 8 experts, M=4096 N=2048, K segments ~ Multinomial(16384) "
                   "padded to 128, 1x128 scales along K, results accumulated into the FP32 C [8,4096,2048] in place "
                   "(D is C)")

    def __init__(self, torch, fg, seed):
        import numpy as np
        import workloads
        self.torch, self.fg = torch, fg
        g, m, n = 8, 4096, 2048
        ks_true = workloads.rng(seed).multinomial(16384, [1.0 / g] * g)
        ks = (ks_true + 127) // 128 * 128
        k_total = int(ks.sum())
        xa = torch.zeros((k_total, m), dtype=torch.float32, device="cuda")
        xb = torch.zeros((k_total, n), dtype=torch.float32, device="cuda")
        off = 0
        for e in range(g):
            t = int(ks_true[e])
            xa[off:off + t] = workloads.device_normal(seed + 10 + e, (t, m))
            xb[off:off + t] = workloads.device_normal(seed + 30 + e, (t, n))
            off += int(ks[e])
        self.a = torch.empty((k_total, m), dtype=torch.uint8, device="cuda")
        self.sfa = torch.zeros((cdiv(k_total, 512), align4(m)), dtype=torch.int32, device="cuda")
        self.b = torch.empty((k_total, n), dtype=torch.uint8, device="cuda")
        self.sfb = torch.zeros((cdiv(k_total, 512), align4(n)), dtype=torch.int32, device="cuda")
        fg.quantize_1x128_cols(xa, self.a, self.sfa)
        fg.quantize_1x128_cols(xb, self.b, self.sfb)
        del xa, xb
        self.ks = torch.from_numpy(ks.astype(np.int32)).cuda()
        self.c = workloads.device_normal(seed + 60, (g, m, n))
        self.d = self.c            # the weight gradient accumulates into C itself
        self.flops = 2.0 * m * n * float(ks_true.sum())
        self.bytes = k_total * (m + n) + self.sfa.numel() * 4 + self.sfb.numel() * 4 + 2 * g * m * n * 4
        self.parts = [{"name": "k_grouped", "flops": self.flops, "bytes": self.bytes}]
        torch.cuda.synchronize()

    def launches(self):
        return [lambda: self.fg.k_grouped_fp8_gemm_tn_contiguous(self.a, self.sfa, self.b, self.sfb, self.ks,
                                                                 self.d, c=self.c)]

    def e2e_io(self):
        ins = [(t, t.cpu().pin_memory()) for t in (self.a, self.sfa, self.b, self.sfb, self.ks, self.c)]
        return ins, [(self.d, self.torch.empty_like(self.d, device="cpu").pin_memory())]


class KGroupedSeparate(KGrouped):
    """The K-grouped workload with a separate D (C read, D written): measurement aid."""
    name = "k_grouped_separate_d"
    description = KGrouped.description.replace("results accumulated into the FP32 C [8,4096,2048] in place (D is C)",
                                               "FP32 C [8,4096,2048] added into a separate FP32 D")

    def __init__(self, torch, fg, seed):
        super().__init__(torch, fg, seed)
        self.d = torch.empty_like(self.c)
        torch.cuda.synchronize()


class Prefill(DensePair):
    """The prefill GEMM alone (profiling aid)."""
    name = "prefill"
    description = "dense FP8 NT GEMM M=4096 N=7168 K=2048, FP32 C accumulated into FP32 D"
    SHAPES = [("prefill", 4096, 7168, 2048)]


class Decode(DensePair):
    """The decode GEMM alone (profiling aid)."""
    name = "decode"
    description = "dense FP8 NT GEMM M=64 N=7168 K=4096, FP32 C accumulated into FP32 D"
    SHAPES = [("decode", 64, 7168, 4096)]


class Small(DensePair):
    """The small dense case: launch latency, not a roofline."""
    name = "small"
    description = "dense FP8 NT GEMM M=128 N=256 K=512, no C, BF16 D"
    SHAPES = [("small", 128, 256, 512)]
    WITH_C = False


class Quant:
    """The quantise/pack kernels on operands of the benchmark GEMMs' sizes: 1x128 row groups
    of an activation x[8192, 7168], 128x128 blocks of a weight w[7168, 2048], 1x128 groups
    along K of a K-grouped operand x[16384, 4096], and MXFP4 (E2M1, 1x32 scales) of the
    expert weights w[32 x 4096, 4096].  HBM-bound streams: one FP32 read, one code write
    and the packed scale words."""
    name = "quant"
    description = ("FP32 -> E4M3 + packed UE8M0 quantisation: 1x128 rows of [8192, 7168], 128x128 "
                   "blocks of [7168, 2048], 1x128 columns of [16384, 4096]; FP32 -> MXFP4 of [32 x 4096, 4096]")

    def __init__(self, torch, fg, seed):
        import workloads
        self.torch, self.fg = torch, fg
        rows_x = workloads.device_normal(seed, (8192, 7168))
        blk_w = workloads.device_normal(seed + 1, (7168, 2048))
        col_x = workloads.device_normal(seed + 2, (16384, 4096))
        mx_w = workloads.device_normal(seed + 3, (32 * 4096, 4096), std=0.02)
        u8, i32 = torch.uint8, torch.int32
        self.items = [
            ("quant_rows", fg.quantize_1x128_rows, rows_x, torch.empty((8192, 7168), dtype=u8, device="cuda"),
             torch.zeros((cdiv(7168, 512), align4(8192)), dtype=i32, device="cuda")),
            ("quant_blocks", fg.quantize_128x128_blocks, blk_w, torch.empty((7168, 2048), dtype=u8, device="cuda"),
             torch.zeros((1, cdiv(2048, 512), align4(cdiv(7168, 128))), dtype=i32, device="cuda")),
            ("quant_cols", fg.quantize_1x128_cols, col_x, torch.empty((16384, 4096), dtype=u8, device="cuda"),
             torch.zeros((cdiv(16384, 512), align4(4096)), dtype=i32, device="cuda")),
            ("quant_mxfp4", fg.quantize_mxfp4, mx_w, torch.empty((32 * 4096, 2048), dtype=u8, device="cuda"),
             torch.zeros((4096 // 128, align4(32 * 4096)), dtype=i32, device="cuda")),
        ]
        self.parts = [{"name": nm, "flops": 0.0, "bound": "hbm",
                       "bytes": x.numel() * 4 + q.numel() + sf.numel() * 4} for nm, _f, x, q, sf in self.items]
        torch.cuda.synchronize()

    def launches(self):
        return [lambda f=f, x=x, q=q, sf=sf: f(x, q, sf) for _nm, f, x, q, sf in self.items]

    def e2e_io(self):
        ins = [(x, x.cpu().pin_memory()) for _nm, _f, x, _q, _sf in self.items]
        outs = [(t, self.torch.empty_like(t, device="cpu").pin_memory())
                for _nm, _f, _x, q, sf in self.items for t in (q, sf)]
        return ins, outs


class Fp4DensePair(DensePair):
    """The dense pair with FP4 weights (the FP8 x FP4 GEMM): B quantised by the library's
    MXFP4 quantiser to E2M1 codes with one UE8M0 scale per 32 K elements of a row."""
    name = "fp4_dense_pair"
    description = ("dense FP8 x FP4 NT GEMM pair: prefill M=4096 N=7168 K=2048 + decode M=64 N=7168 K=4096; "
                   "A 1x128 UE8M0, B E2M1 with 1x32 UE8M0 scales; FP32 C accumulated into FP32 D")
    PREFIX = "fp4_"

    @staticmethod
    def make_weights(torch, fg, xb, n, k):
        b = torch.empty((n, k // 2), dtype=torch.uint8, device="cuda")
        sfb = torch.zeros((k // 128, align4(n)), dtype=torch.int32, device="cuda")
        fg.quantize_mxfp4(xb, b, sfb)
        return b, sfb

    def launches(self):
        return [lambda p=p: self.fg.fp8_fp4_gemm_nt(p["a"], p["sfa"], p["b"], p["sfb"], p["d"], c=p["c"])
                for p in self.parts]


class Fp4Prefill(Fp4DensePair):
    name = "fp4_prefill"
    description = "dense FP8 x FP4 NT GEMM M=4096 N=7168 K=2048, FP32 C accumulated into FP32 D"
    SHAPES = [("prefill", 4096, 7168, 2048)]


class Fp4Decode(Fp4DensePair):
    name = "fp4_decode"
    description = "dense FP8 x FP4 NT GEMM M=64 N=7168 K=4096, FP32 C accumulated into FP32 D"
    SHAPES = [("decode", 64, 7168, 4096)]


class Fp4Contiguous(Contiguous):
    name = "fp4_contiguous"
    description = ("M-grouped contiguous FP8 x FP4 NT GEMM: the contiguous configuration (32 experts, N=4096 "
                   "K=4096, BF16 D) with E2M1 expert weights and 1x32 UE8M0 scales")

    @staticmethod
    def make_expert_weights(torch, fg, seed, g, n, k):
        """Per expert: N(0, 0.02^2) draws, MXFP4 by the library's quantiser."""
        import workloads
        b = torch.empty((g, n, k // 2), dtype=torch.uint8, device="cuda")
        sfb = torch.zeros((g, k // 128, align4(n)), dtype=torch.int32, device="cuda")
        for e in range(g):
            xb = workloads.device_normal(seed + 100 + e, (1, n, k), std=0.02)
            fg.quantize_mxfp4(xb, b[e:e + 1], sfb[e:e + 1])
        return b, sfb

    def launches(self):
        return [lambda: self.fg.m_grouped_fp8_fp4_gemm_nt_contiguous(self.a, self.sfa, self.b, self.sfb,
                                                                     self.m_indices, self.d)]


class Fp4Masked(Masked):
    name = "fp4_masked"
    description = ("M-grouped masked FP8 x FP4 NT GEMM: the masked configuration (32 experts x 256 rows, N=4096 "
                   "K=2048, BF16 D) with E2M1 expert weights and 1x32 UE8M0 scales")
    make_expert_weights = staticmethod(Fp4Contiguous.make_expert_weights)

    def launches(self):
        return [lambda: self.fg.m_grouped_fp8_fp4_gemm_nt_masked(self.a, self.sfa, self.b, self.sfb, self.masked_m,
                                                                 self.d, expected_m=self.expected_m)]


class _PrefillLayout(Prefill):
    """The prefill GEMM with its operands stored in another layout (same values, same
    bytes and FLOPs): A as [K, M] for a leading T, B as [K, N] for a trailing N."""
    LAYOUT = "nn"

    def __init__(self, torch, fg, seed):
        super().__init__(torch, fg, seed)
        p = self.parts[0]
        if self.LAYOUT[0] == "t":
            p["a"] = p["a"].t().contiguous()
        if self.LAYOUT[1] == "n":
            p["b"] = p["b"].t().contiguous()
        torch.cuda.synchronize()

    def launches(self):
        fn = getattr(self.fg, "fp8_gemm_" + self.LAYOUT)
        return [lambda p=p: fn(p["a"], p["sfa"], p["b"], p["sfb"], p["d"], c=p["c"]) for p in self.parts]


class PrefillNN(_PrefillLayout):
    name, LAYOUT = "prefill_nn", "nn"
    description = "dense FP8 NN GEMM (B stored [K,N]) M=4096 N=7168 K=2048, FP32 C accumulated into FP32 D"


class PrefillTN(_PrefillLayout):
    name, LAYOUT = "prefill_tn", "tn"
    description = "dense FP8 TN GEMM (A [K,M], B [K,N]) M=4096 N=7168 K=2048, FP32 C accumulated into FP32 D"


class PrefillTT(_PrefillLayout):
    name, LAYOUT = "prefill_tt", "tt"
    description = "dense FP8 TT GEMM (A stored [K,M]) M=4096 N=7168 K=2048, FP32 C accumulated into FP32 D"


class ContiguousSwiGLU(Contiguous):
    """The contiguous workload as the MoE gate-up GEMM with the fused SwiGLU + FP8
    requantisation epilogue: B [32, 2 x 2048, 4096] (gate rows, then up rows), output
    q [M_total, 2048] E4M3 + packed UE8M0 scales (the down projection's A operand)."""
    name = "contiguous_swiglu"
    description = ("M-grouped contiguous FP8 gate-up GEMM with fused SwiGLU + per-1x128 E4M3 requantisation: "
                   "32 experts (top-6 of 8192 tokens, experts 0-31, 128-row padded segments), I=2048 (B 2I=4096 "
                   "rows), K=4096; output E4M3 [M_total, 2048] + UE8M0 scales")

    def __init__(self, torch, fg, seed):
        super().__init__(torch, fg, seed)
        m_total, inter = self.a.shape[0], self.b.shape[1] // 2
        self.q = torch.empty((m_total, inter), dtype=torch.uint8, device="cuda")
        self.sfq = torch.zeros((cdiv(inter, 512), align4(m_total)), dtype=torch.int32, device="cuda")
        k, nv = self.a.shape[1], self.nv
        self.bytes = (nv * k + self.used * self.b[0].numel() + self.sfa.numel() * 4 + self.sfb.numel() * 4
                      + nv * inter + nv * (inter // 128) + m_total * 4)
        self.parts = [{"name": self.name, "flops": self.flops, "bytes": self.bytes}]
        del self.d
        torch.cuda.synchronize()

    def launches(self):
        return [lambda: self.fg.m_grouped_fp8_gemm_nt_contiguous_swiglu(self.a, self.sfa, self.b, self.sfb,
                                                                        self.m_indices, self.q, self.sfq)]

    def e2e_io(self):
        ins = [(t, t.cpu().pin_memory()) for t in (self.a, self.sfa, self.b, self.sfb, self.m_indices)]
        return ins, [(t, self.torch.empty_like(t, device="cpu").pin_memory()) for t in (self.q, self.sfq)]


class Fp4ContiguousSwiGLU(ContiguousSwiGLU):
    """The fused gate-up GEMM with FP4 expert weights (the Mega MoE's linear 1 in FP8 x FP4,
    then SwiGLU and the requantisation for linear 2)."""
    name = "fp4_contiguous_swiglu"
    description = ("M-grouped contiguous FP8 x FP4 gate-up GEMM with fused SwiGLU + per-1x128 E4M3 "
                   "requantisation: the contiguous_swiglu configuration with E2M1 expert weights and 1x32 "
                   "UE8M0 scales")
    make_expert_weights = staticmethod(Fp4Contiguous.make_expert_weights)

    def launches(self):
        return [lambda: self.fg.m_grouped_fp8_fp4_gemm_nt_contiguous_swiglu(self.a, self.sfa, self.b, self.sfb,
                                                                            self.m_indices, self.q, self.sfq)]


class MoeMlp(ContiguousSwiGLU):
    """The MoE expert MLP of the contiguous configuration on one GPU: linear 1 (gate-up, I =
    2048, K = 4096) with the fused SwiGLU + E4M3 requantisation, then linear 2 (the down
    projection, [32, 4096, 2048] weights) on its output, BF16 D.  One step = both GEMMs."""
    name = "moe_mlp"
    description = ("MoE expert MLP, contiguous layout (32 experts, top-6 of 8192 tokens): gate-up GEMM with fused "
                   "SwiGLU + E4M3 requantisation (I=2048, K=4096), then the down projection (N=4096, K=2048), BF16 D")

    def __init__(self, torch, fg, seed):
        super().__init__(torch, fg, seed)
        g, inter = self.b.shape[0], self.q.shape[1]
        hidden = self.a.shape[1]
        self.w2, self.sfw2 = self.make_expert_weights(torch, fg, seed + 5000, g, hidden, inter)
        m_total = self.a.shape[0]
        self.d = torch.empty((m_total, hidden), dtype=torch.bfloat16, device="cuda")
        nv = self.nv
        down_flops = 2.0 * nv * hidden * inter
        down_bytes = (nv * inter + self.sfq.numel() * 4 + self.used * self.w2[0].numel() + self.sfw2.numel() * 4
                      + nv * hidden * 2 + m_total * 4)
        self.parts = [self.parts[0], {"name": self.name + "_down", "flops": down_flops, "bytes": down_bytes}]
        torch.cuda.synchronize()

    def down(self):
        self.fg.m_grouped_fp8_gemm_nt_contiguous(self.q, self.sfq, self.w2, self.sfw2, self.m_indices, self.d)

    def launches(self):
        return super().launches() + [self.down]

    def e2e_io(self):
        ins = [(t, t.cpu().pin_memory()) for t in (self.a, self.sfa, self.b, self.sfb, self.w2, self.sfw2,
                                                     self.m_indices)]
        return ins, [(self.d, self.torch.empty_like(self.d, device="cpu").pin_memory())]


class Fp4MoeMlp(MoeMlp):
    """The MoE expert MLP with FP4 (MXFP4) weights in both GEMMs."""
    name = "fp4_moe_mlp"
    description = ("MoE expert MLP in FP8 x FP4: the moe_mlp configuration with E2M1 expert weights and 1x32 "
                   "UE8M0 scales in both GEMMs")
    make_expert_weights = staticmethod(Fp4Contiguous.make_expert_weights)

    def launches(self):
        return Fp4ContiguousSwiGLU.launches(self) + [self.down]

    def down(self):
        self.fg.m_grouped_fp8_fp4_gemm_nt_contiguous(self.q, self.sfq, self.w2, self.sfw2, self.m_indices, self.d)


class MqaLogits:
    """Lightning-indexer MQA logits (non-paged): 4096 query tokens x 4096 kv tokens, causal
    ranges (token i sees kv [0, i]), 64 heads, D = 128, clean_logits; FP32 out [4096, 4096].
    Tensor-bound: 137 GFLOP of FP8 products against ~100 MB of traffic."""
    name = "mqa_logits"
    description = ("FP8 MQA logits: S=4096 query x T=4096 kv tokens, causal ranges, H=64 heads, D=128, "
                   "kv per-token FP32 scales, clean_logits; FP32 logits [4096, 4096]")
    S, T, H, D = 4096, 4096, 64, 128

    def __init__(self, torch, fg, seed):
        import workloads
        self.torch, self.fg = torch, fg
        s_len, t_len, heads, dim = self.S, self.T, self.H, self.D
        xq = workloads.device_normal(seed, (s_len * heads, dim))
        self.q = torch.empty((s_len * heads, dim), dtype=torch.uint8, device="cuda")
        sfq = torch.zeros((cdiv(dim, 512), align4(s_len * heads)), dtype=torch.int32, device="cuda")
        fg.quantize_1x128_rows(xq, self.q, sfq)     # E4M3 codes; the per-row scales are not used
        self.q = self.q.view(s_len, heads, dim)
        xk = workloads.device_normal(seed + 1, (t_len, dim))
        self.kv = torch.empty((t_len, dim), dtype=torch.uint8, device="cuda")
        sfk = torch.zeros((1, align4(t_len)), dtype=torch.int32, device="cuda")
        fg.quantize_1x128_rows(xk, self.kv, sfk)
        self.kv_sf = torch.ldexp(torch.ones(t_len, device="cuda"),
                                 (sfk[0, :t_len] & 0xFF).to(torch.int32) - 127).float()
        del xq, xk
        self.w = workloads.device_normal(seed + 2, (s_len, heads))
        self.ks = torch.zeros(s_len, dtype=torch.int32, device="cuda")
        self.ke = torch.arange(1, s_len + 1, dtype=torch.int32, device="cuda")
        self.out = torch.empty((s_len, t_len), dtype=torch.float32, device="cuda")
        pairs = s_len * (s_len + 1) // 2
        self.flops = 2.0 * pairs * heads * dim
        self.bytes = s_len * heads * dim + t_len * dim + t_len * 4 + s_len * heads * 4 + 2 * s_len * 4 + s_len * t_len * 4
        self.parts = [{"name": "mqa_logits", "flops": self.flops, "bytes": self.bytes, "bound": "tensor"}]
        torch.cuda.synchronize()

    def launches(self):
        return [lambda: self.fg.fp8_mqa_logits(self.q, self.kv, self.kv_sf, self.w, self.ks, self.ke, self.out)]

    def e2e_io(self):
        ins = [(t, t.cpu().pin_memory()) for t in (self.q, self.kv, self.kv_sf, self.w, self.ks, self.ke)]
        return ins, [(self.out, self.torch.empty_like(self.out, device="cpu").pin_memory())]


class ContiguousNN(Contiguous):
    """The contiguous workload with each expert's weights stored [K, N]."""
    name = "contiguous_nn"
    description = Contiguous.description.replace("contiguous FP8 NT GEMM", "contiguous FP8 NN GEMM (B [G,K,N])")

    def __init__(self, torch, fg, seed):
        super().__init__(torch, fg, seed)
        self.b = self.b.transpose(1, 2).contiguous()
        torch.cuda.synchronize()

    def launches(self):
        return [lambda: self.fg.m_grouped_fp8_gemm_nn_contiguous(self.a, self.sfa, self.b, self.sfb,
                                                                 self.m_indices, self.d)]


WORKLOADS = {w.name: w for w in (DensePair, Prefill, Decode, Small, Contiguous, Masked, KGrouped, KGroupedSeparate, Quant, PrefillNN,
                                 PrefillTN, PrefillTT, ContiguousNN, ContiguousSwiGLU, MqaLogits, Fp4DensePair,
                                 Fp4Prefill, Fp4Decode, Fp4Contiguous, Fp4Masked, Fp4ContiguousSwiGLU, MoeMlp,
                                 Fp4MoeMlp)}

# The benchmark configurations beside the headline pair (recorded in config.kernels of
# the default run): (configuration number, workload).
# (configuration number, or the scope row for the quantisers, which no configuration names)
OTHER_CONFIGS = [(0, "small"), (2, "contiguous"), (3, "masked"), (4, "k_grouped"), ("NEXT-1", "quant"),
                 ("NEXT-4", "fp4_dense_pair"), ("NEXT-4", "fp4_contiguous"), ("NEXT-4", "fp4_masked")]
NOMINAL_HBM_GBS = 8000.0        # the stated HBM roof (about 8 TB/s)
NOMINAL_FP8_TFLOPS = 4500.0     # the stated dense FP8 tensor roof (about 4.5 PFLOP/s)
MIN_TIMED_SECONDS = 0.5         # repeat the --steps pass until the timed region lasts this long
REFERENCE_BUDGET_S = 150.0      # CPU seconds the reference arm may spend on its steps


# ------------------------------------------------------------------- CPU oracle arm
def time_oracle(items, min_seconds=10.0, max_reps=8):
    reps, flops, t0 = 0, 0.0, time.perf_counter()
    while reps < max_reps:
        for fn, f in items:
            fn()
            flops += f
        reps += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    return flops, time.perf_counter() - t0, reps


def run_reference(args):
    """The reference arm: the CPU oracle timed on the machine's host cores.  Each step is one
    full dense-pair step (every output of both GEMMs, the same work as the GPU arm's step
    and as ``cpu_baseline``) when --warmup + --steps of them fit in REFERENCE_BUDGET_S;
    otherwise each step is the bounded sample ``oracle_sub_step`` (first rows x columns of
    each GEMM) so that the run still ends within a few minutes."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    if args.workload != "dense_pair":
        print(json.dumps({"impl": "reference", "unavailable": "the CPU oracle arm covers the dense_pair workload"}))
        return 0
    cores = len(os.sched_getaffinity(0))
    items, sample = DensePair.oracle_full_step()
    t0 = time.perf_counter()
    for fn, _f in items:                     # first warm-up step, also the size estimate
        fn()
    t_full = time.perf_counter() - t0
    if (args.warmup - 1 + args.steps) * t_full > REFERENCE_BUDGET_S:
        # the sample's rows and columns both shrink (the oracle dequantises the columns'
        # weights on every call), to about `frac` of a full step's work
        frac = REFERENCE_BUDGET_S / ((args.warmup + args.steps) * t_full)
        side = math.sqrt(frac)
        items, sample = DensePair.oracle_sub_step(rows=max(32, int(4096 * side)),
                                                  cols=max(256, int(7168 * side) // 128 * 128))
        warm_left = args.warmup
    else:
        warm_left = args.warmup - 1
    for _ in range(warm_left):
        for fn, _f in items:
            fn()
    flops, t0 = 0.0, time.perf_counter()
    for _ in range(args.steps):
        for fn, f in items:
            fn()
            flops += f
    t = time.perf_counter() - t0
    value = flops / t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: seeded numpy N(0,1) draws quantised by the oracle",
            "config": {"workload": DensePair.description},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------ GPU arm
def max_over_ranks(torch, dist, value: float, device: str) -> float:
    """The largest of every rank's `value` (the slowest rank sets a whole-job time);
    `value` itself on one process."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank_step: float, step_ms: float) -> float:
    """Aggregate throughput: every rank does one step of `flops_per_rank_step` in at most
    `step_ms` (the max over ranks)."""
    return world * flops_per_rank_step / (step_ms * 1e-3) / 1e12


def kernel_entry(p: dict, us: float, peaks: dict) -> dict:
    """Per-kernel record: time, throughput and its fraction of each roof (the stated
    nominal roofs first, the measured ones second)."""
    t = us * 1e-6
    tflops, gbs = p["flops"] / t / 1e12, p["bytes"] / t / 1e9
    fp8_measured = peaks["bf16_tflops"] * FP8_OVER_BF16
    t_roof_nominal = max(p["flops"] / (NOMINAL_FP8_TFLOPS * 1e12), p["bytes"] / (NOMINAL_HBM_GBS * 1e9))
    t_roof_measured = max(p["flops"] / (fp8_measured * 1e12), p["bytes"] / (peaks["hbm_gbs"] * 1e9))
    return {
        "us_per_launch": round(us, 2), "tflops": round(tflops, 1), "hbm_gbs": round(gbs, 1),
        "algorithmic_bytes": p["bytes"], "flops": p["flops"],
        "bound": "tensor" if p["flops"] / fp8_measured / 1e12 > p["bytes"] / peaks["hbm_gbs"] / 1e9 else "hbm",
        "frac_of_roof_nominal": round(t_roof_nominal / t, 3),
        "frac_of_hbm_nominal": round(gbs / NOMINAL_HBM_GBS, 3),
        "frac_of_fp8_tensor_nominal": round(tflops / NOMINAL_FP8_TFLOPS, 3),
        "frac_of_roof": round(t_roof_measured / t, 3),
        "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3),
        "frac_of_fp8_tensor": round(tflops / fp8_measured, 3),
    }


def time_steps(torch, launches, steps, flush, stream, per_kernel):
    """One timed pass of `steps` steps, L2 flushed (outside the events) before each when
    `flush` is a buffer (None: no flush).
    per_kernel=False: events at the step boundaries only, returns the mean step time (ms).
    per_kernel=True: an event after every launch, returns the mean time of each (ms)."""
    nl = len(launches)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1 if per_kernel else 2)]
          for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.fill_(1)
        ev[i][0].record(stream)
        for j, fn in enumerate(launches):
            fn()
            if per_kernel:
                ev[i][j + 1].record(stream)
        if not per_kernel:
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    if per_kernel:
        return [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)) / steps for j in range(nl)]
    return sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)) / steps


def run_gpu(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import moe_fp8_e4m3_gb300 as fg

    wl = WORKLOADS[args.workload](torch, fg, args.seed + 7919 * rank)
    launches = wl.launches()
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")

    def flush_for(work):
        """The L2 rule of a workload: flush before every step (a write of 2x L2) unless one
        step reads and writes more than twice the L2 size by itself."""
        step_bytes = sum(p["bytes"] for p in work.parts)
        if args.l2 == "flush" or (args.l2 == "auto" and step_bytes < 2 * l2):
            return flush_buf, "flushed before every timed step (write of 2x L2)"
        return None, (f"not flushed: one step moves {step_bytes / 1e6:.0f} MB, more than twice the "
                      f"{l2 / 1e6:.0f} MB L2")

    flush, l2_note = flush_for(wl)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        if flush is not None:
            flush.fill_(1)
        for fn in launches:
            fn()
    barrier()
    # pass length estimate (warm-up steps, flush included) -> passes for the timed region
    t_est = time.perf_counter()
    for _ in range(min(args.steps, 20)):
        if flush is not None:
            flush.fill_(1)
        for fn in launches:
            fn()
    barrier()
    per_step_s = (time.perf_counter() - t_est) / min(args.steps, 20)
    passes = max(1, min(200, math.ceil(MIN_TIMED_SECONDS / max(per_step_s * args.steps, 1e-9))))
    st, detail = fg.get_device_error()
    if st != 0:
        raise RuntimeError(f"device status {st} ({detail:#x}) during warm-up")

    nl = len(launches)
    sampler = ClockSampler(local)
    time.sleep(0.3)
    barrier()
    t_wall0 = time.time()
    # pass 1 (x passes): step time, events at the step boundaries only
    step_runs = []
    for _ in range(passes):
        barrier()
        step_runs.append(time_steps(torch, launches, args.steps, flush, stream, False))
    barrier()
    # pass 2 (x passes): per-kernel durations, an event after every GEMM
    kernel_runs = []
    for _ in range(passes):
        kernel_runs.append(time_steps(torch, launches, args.steps, flush, stream, True))
    barrier()
    t_wall1 = time.time()
    time.sleep(0.15)
    sampler.stop()
    st, detail = fg.get_device_error()
    if st != 0:
        raise RuntimeError(f"device status {st} ({detail:#x}) in the timed region")

    per_kernel = [sum(r[j] for r in kernel_runs) / passes for j in range(nl)]     # ms, mean per launch
    step_ms = sum(step_runs) / passes
    step_ms = max_over_ranks(torch, dist, step_ms, "cuda")
    flops_step = sum(p["flops"] for p in wl.parts)
    value = whole_job_tflops(world, flops_step, step_ms)
    gpu_launches = 2 * nl * args.steps * passes

    # ---- the other benchmark configurations (default run only): each timed alone on the
    # same rules (the L2 rule above, --warmup untimed steps, one pass of --steps)
    peaks = load_peaks()
    kernels = {}
    for j, p in enumerate(wl.parts):
        kernels[p["name"]] = dict(kernel_entry(p, per_kernel[j] * 1e3, peaks), config=1) \
            if args.workload == "dense_pair" else kernel_entry(p, per_kernel[j] * 1e3, peaks)
    if args.workload == "dense_pair" and not args.no_other_configs:
        for cfg_no, name in OTHER_CONFIGS:
            owl = WORKLOADS[name](torch, fg, args.seed + 101 * (cfg_no if isinstance(cfg_no, int) else 9) + 7919 * rank)
            ol = owl.launches()
            oflush, onote = flush_for(owl)
            for _ in range(args.warmup):
                if oflush is not None:
                    oflush.fill_(1)
                for fn in ol:
                    fn()
            ot = time_steps(torch, ol, args.steps, oflush, stream, True)
            gpu_launches += len(ol) * args.steps
            st, detail = fg.get_device_error()
            if st != 0:
                raise RuntimeError(f"device status {st} ({detail:#x}) in configuration {cfg_no}")
            for j, p in enumerate(owl.parts):
                e = kernel_entry(p, ot[j] * 1e3, peaks)
                e["config"] = cfg_no
                e["workload"] = owl.description
                e["l2"] = onote
                if cfg_no == 0:
                    e["note"] = "launch-latency case: report the time, not a roofline fraction"
                kernels[p["name"]] = e
            del owl, ol
            torch.cuda.empty_cache()

    # ---- end to end through the public API with host buffers
    # Every step copies its inputs host -> device (pinned), runs the GEMMs and reads the
    # results back device -> host; the two directions use separate copy engines.
    # (Spreading the input copies over several streams measured no faster: the host link,
    # not one DMA queue, sets the input rate.)
    e2e_steps = max(3, min(args.steps, 50))
    out_stream = torch.cuda.Stream()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if hasattr(wl, "e2e_double"):
        # Double-buffered: step i uses device set i % 2, so step i+1's input copies (their own
        # stream) run beside step i's GEMMs and step i-1's read-back; a set is refilled only
        # after the GEMMs of the step that used it two steps before, and its D is overwritten
        # only after that step's read-back.  Time: step 2's first input copy to the last
        # read-back, / steps.
        bind, io = wl.e2e_double()
        ins, outs = io[0]
        in_stream = torch.cuda.Stream()
        comp = [None, None]
        out_done = [None, None]
        for i in range(e2e_steps + 2):
            k = i % 2
            if comp[k] is not None:
                in_stream.wait_event(comp[k])
            if i == 2:
                t_start.record(in_stream)
            with torch.cuda.stream(in_stream):
                for dt, ht in io[k][0]:
                    dt.copy_(ht, non_blocking=True)
            landed = torch.cuda.Event()
            landed.record(in_stream)
            stream.wait_event(landed)
            if out_done[k] is not None:
                stream.wait_event(out_done[k])
            bind(k)
            for fn in launches:
                fn()
            comp[k] = torch.cuda.Event()
            comp[k].record(stream)
            out_stream.wait_event(comp[k])
            with torch.cuda.stream(out_stream):
                for dt, ht in io[k][1]:
                    ht.copy_(dt, non_blocking=True)
                out_done[k] = torch.cuda.Event()
                out_done[k].record(out_stream)
        t_end.record(out_stream)
        torch.cuda.synchronize()
        bind(0)
        e2e_overlap = ("double-buffered device inputs and outputs: step i+1's host-to-device copies run "
                       "beside step i's GEMMs and step i-1's device-to-host read-back")
    else:
        # Step i's read-back runs on a second stream while step i+1's inputs go in; step
        # i+1's GEMMs wait for step i's read-back (they overwrite D) and step i+1's input
        # copies wait for step i's GEMMs (stream order).
        ins, outs = wl.e2e_io()
        out_done = None
        for i in range(e2e_steps + 2):
            if i == 2:
                stream.wait_stream(out_stream)
                t_start.record(stream)
            for dt, ht in ins:
                dt.copy_(ht, non_blocking=True)
            if out_done is not None:
                stream.wait_event(out_done)
            for fn in launches:
                fn()
            computed = torch.cuda.Event()
            computed.record(stream)
            out_stream.wait_event(computed)
            with torch.cuda.stream(out_stream):
                for dt, ht in outs:
                    ht.copy_(dt, non_blocking=True)
                out_done = torch.cuda.Event()
                out_done.record(out_stream)
        stream.wait_event(out_done)
        t_end.record(stream)
        torch.cuda.synchronize()
        e2e_overlap = "step i's device-to-host read-back runs beside step i+1's host-to-device copies"
    h2d = sum(t.numel() * t.element_size() for t, _ in ins)
    d2h = sum(t.numel() * t.element_size() for t, _ in outs)
    e2e_ms = t_start.elapsed_time(t_end) / e2e_steps
    e2e_ms = max_over_ranks(torch, dist, e2e_ms, "cuda")
    e2e_value = whole_job_tflops(world, flops_step, e2e_ms)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    dom = max(range(nl), key=lambda j: per_kernel[j])
    part = wl.parts[dom]
    achieved = part["bytes"] / (per_kernel[dom] * 1e-3) / 1e9
    traffic = recorded_traffic(wl.name, part["name"])
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)",
        "data": "synthetic: seeded N(0,1) draws (torch generator on the GPU) quantised by the library's "
                "UE8M0 quantise kernels",
        "config": {"workload": wl.description, "l2": l2_note,
                   "replicas": world, "pdl": fg.get_pdl(), "passes": passes,
                   "timing": f"{passes} back-to-back passes of --steps steps each, averaged; step: events at "
                             "step boundaries only; kernels: a second set of passes with an event after every "
                             "GEMM; other configurations: one pass each, an event after every launch",
                   "roofs": {"nominal": {"hbm_gbs": NOMINAL_HBM_GBS, "fp8_tflops": NOMINAL_FP8_TFLOPS},
                             "measured": {"hbm_gbs": peaks["hbm_gbs"], "fp8_tflops": round(fp8_peak, 1),
                                          "source": peaks["source"]}},
                   "kernels": kernels},
        "roofline": ({"bound": "hbm", "kernel": part["name"], "achieved": round(achieved, 1),
                      "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                      "traffic": traffic, "algorithmic_bytes_per_launch": part["bytes"],
                      "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)"}
                     if part.get("bound", "hbm") == "hbm" else
                     {"bound": "tensor", "kernel": part["name"],
                      "achieved": round(part["flops"] / (per_kernel[dom] * 1e-3) / 1e12, 1),
                      "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                      "frac": round(part["flops"] / (per_kernel[dom] * 1e-3) / 1e12 / fp8_peak, 4),
                      "traffic": traffic, "algorithmic_flops_per_launch": part["flops"],
                      "peak_source": f"{peaks['source']} bf16 burst x {FP8_OVER_BF16} (nominal fp8/bf16 ratio)"}),
        "roofline_tensor": {"kernel": part["name"],
                            "achieved": round(part["flops"] / (per_kernel[dom] * 1e-3) / 1e12, 1),
                            "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                            "frac": round(part["flops"] / (per_kernel[dom] * 1e-3) / 1e12 / fp8_peak, 4),
                            "peak_source": f"{peaks['source']} bf16 burst x {FP8_OVER_BF16} (nominal fp8/bf16 ratio)"},
        "clocks": sampler.summary(t_wall0, t_wall1),
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "overlap": e2e_overlap},
        "gpu_launches": gpu_launches,
        "cpu_baseline": None,
    }
    if world == 1 and not args.no_cpu_baseline and args.workload == "dense_pair":
        items, sample = DensePair.oracle_full_step()
        f, dt, reps = time_oracle(items)
        line["cpu_baseline"] = {"value": round(f / dt / 1e12, 5), "unit": "TFLOP/s",
                                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": f"{sample}, {reps} repetition(s), {dt:.1f} s"}
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["fg", "reference"], default="fg")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="dense_pair")
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2", choices=["auto", "flush", "none"], default="auto",
                    help="auto: flush L2 before every step unless one step moves more than twice L2")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="time only the headline pair (skip configurations 0, 2, 3 and 4)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
