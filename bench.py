"""Throughput of the gapped varlen attention forward on GB300.

One step = one pass of the whole hot path over one batch of synthetic input: the
forward launch(es) and, for partitioned workloads, the LSE merge (for the
``long_replay_bwd`` workload: the backward, dQ / dK / dV, of the long replay). The default workload
is the long joint video + LiDAR replay (4 segments x 32768 query rows, 65536 keys each,
seeded used fractions; Hq=32, Hkv=8, d=128, bf16), the largest single-GPU workload.

Metric: useful TFLOP/s over used rows (4 * d * Hq * sum_b used_q[b] * used_k[b] per
launch) divided by the device time per step (CUDA events on the launching stream).

  python bench.py [--gpus N --steps K --warmup W] [--impl gva|reference] [--workload NAME]

With torchrun (N > 1) every rank runs its own copy of the workload on its own GPU (the
path shards by independent problems; there is no data-path collective), and the value
is the total work of all ranks over the slowest rank's time.
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
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "gapped-varlen attn fwd TFLOP/s (used rows) & % of GB300 BF16 peak; ms/launch"
UNIT = "TFLOP/s"
CSRC = os.path.join(ROOT, "gapped_varlen_attention_gb300", "csrc")
# DRAM bytes per launch of each workload's dominant kernel, as ncu measured them, with
# the hash of the kernel sources they were measured on (written by hand from ncu output)
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "dram_traffic.json")
# the sources behind each timed kernel: its .cu file and the device headers it includes
KERNEL_SOURCES = {
    "gva_fwd_kernel": ["gva_fwd.cu", "gva_device_common.cuh", "sm103_ptx.cuh", "gva_internal.h"],
    "gva_backward": ["gva_bwd.cu", "gva_device_common.cuh", "sm103_ptx.cuh", "gva_internal.h"],
    "gva_lse_merge_kernel": ["gva_merge.cu", "gva_device_common.cuh", "sm103_ptx.cuh", "gva_internal.h"],
}
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


# --------------------------------------------------------------------------------------
# Workloads: each returns (description, setup(device) -> step callable, flops per step,
# launches per step, host/device byte counts).
# --------------------------------------------------------------------------------------

def _describe(g):
    return {"segments": g.num_segments, "total_q": g.total_q, "total_k": g.total_k,
            "used_q": [int(x) for x in g.used_q], "used_k": [int(x) for x in g.used_k],
            "heads_q": g.num_heads_q, "heads_kv": g.num_heads_kv, "head_dim": g.head_dim}


LABELS = {
    "long_replay": ("long joint video+LiDAR replay: 4 segments x 32768 q rows (used 60-100%) x 65536 keys "
                    "(used 50-100%), Hq=32, Hkv=8, d=128, bf16, non-causal"),
    "long_replay_small": "reduced long replay (profiling): 2 segments x 8192 q rows x 32768 keys, Hq=32, Hkv=8",
    "cfg_text_cross": "CFG B=2 text cross-attention: 2 x 4096 q rows, text keys 700 / 20 of 1024, Hq=16, Hkv=8",
    "multiview_causal": "multiview causal gapped replay: 7 segments, 2 visibility partitions + FP32 LSE merge",
    "multiview_fused": "multiview causal gapped replay: 7 segments, 2 visibility partitions fused in one launch",
    "multiview_blockcausal": ("multiview causal gapped replay: 7 segments, block-causal masking with 512-token "
                              "frames in one launch (FLOPs count visible keys only)"),
    "long_replay_bwd": ("backward (dQ, dK, dV) of the long joint video+LiDAR replay: 4 segments x 32768 q rows "
                        "(used 60-100%) x 65536 keys (used 50-100%), Hq=32, Hkv=8, d=128, bf16; FLOPs = 2.5 x "
                        "the forward's (five used-row products)"),
    "multiview_fused_bwd": ("backward of the multiview causal gapped replay with its 2 visibility partitions as "
                            "two key ranges per segment of one plan"),
    "multiview_blockcausal_bwd": ("backward of the multiview causal gapped replay with 512-token block-causal "
                                  "masking (FLOPs: 2.5 x the visible-key forward FLOPs)"),
    "long_replay_small_bwd": "backward of the reduced long replay (profiling): 2 segments x 8192 q rows x 32768 keys",
    "lse_merge_union": ("text + video LSE merge: 8192 q rows in 10 segments, each attending its own 1024 text and "
                        "16384 video keys as 2 launches (FP32 partials) + FP32 LSE merge, one segment's text "
                        "partition empty; Hq=Hkv=24, d=128"),
    "lse_merge": ("the FP32 LSE merge alone on the text + video workload's partials: 8192 q rows in 10 "
                  "segments, 2 FP32 partitions (one segment's text partition keyless), bf16 output, Hq=24, d=128"),
    "tiny": "tiny: 3 segments, Hq=4, Hkv=2, d=64",
}
WORKLOADS = tuple(LABELS)


def spec(name: str):
    """The host-side description of a workload, shared by both arms: its geometries
    (one per forward launch), the merged geometry of partitioned ones (`parts`), the
    geometry and seed its Q / K / V are drawn from, and its options."""
    from gapped_varlen_attention_gb300 import workloads as W
    if name not in LABELS:
        raise SystemExit(f"unknown workload {name}")
    sp = types.SimpleNamespace(name=name, label=LABELS[name], parts=None, ranges=None, causal_block=0,
                               backward=name.endswith("_bwd"), merge_only=False, k_pad_fill=None,
                               part_kv_geoms=None, used_k_parts=None)
    base = name[:-4] if sp.backward else name
    if base in ("long_replay", "long_replay_small"):
        g = W.long_replay() if base == "long_replay" else W.long_replay_small()
        sp.geoms, sp.qkv_geom, sp.seed = [g], g, 1005 if base == "long_replay" else 1006
    elif base == "cfg_text_cross":
        g = W.cfg_text_cross()
        sp.geoms, sp.qkv_geom, sp.seed, sp.k_pad_fill = [g], g, 1002, 0.0
    elif base.startswith("multiview"):
        full, parts = W.multiview_causal()
        sp.qkv_geom, sp.seed = full, 1003
        if base == "multiview_causal":
            sp.geoms, sp.parts = parts, full
        else:
            sp.geoms = [full]
        if base == "multiview_fused":
            sp.ranges = [[(int(p.cu_k[b]), int(p.used_k[b])) for p in parts] for b in range(full.num_segments)]
        if base == "multiview_blockcausal":
            sp.causal_block = 512
    elif base in ("lse_merge_union", "lse_merge"):
        text, video, union, _ = W.lse_merge_union()
        sp.parts, sp.qkv_geom, sp.seed = union, text, 1004
        if base == "lse_merge_union":
            sp.geoms, sp.part_kv_geoms = [text, video], [(text, 1004), (video, 2004)]
        else:
            sp.geoms, sp.merge_only, sp.used_k_parts = [union], True, [text.used_k, video.used_k]
    else:
        g = W.tiny()
        sp.geoms, sp.qkv_geom, sp.seed = [g], g, 1001
    return sp


def spec_input_bytes(sp) -> int:
    """Bytes of the step's device-resident inputs (whole buffers, gap rows included)."""
    qg = sp.parts if sp.parts is not None else sp.geoms[0]
    q = qg.total_q * qg.num_heads_q * qg.head_dim * 2
    lse = qg.num_heads_q * qg.total_q * 4
    if sp.merge_only:
        return len(sp.used_k_parts) * (2 * q + lse)
    kv_geoms = [g for g, _ in sp.part_kv_geoms] if sp.part_kv_geoms is not None else [sp.qkv_geom]
    kv = sum(2 * g.total_k * g.num_heads_kv * g.head_dim * 2 for g in kv_geoms)
    return q + kv + ((2 * q + lse) if sp.backward else 0)


def spec_config(sp, per_step: dict, parallelism: str) -> dict:
    """The `config` object of a bench line: the same for both arms of one workload."""
    geom = sp.parts if sp.parts is not None else sp.geoms[0]
    input_bytes = spec_input_bytes(sp)
    return {"workload": sp.name, "description": sp.label, **_describe(geom), **per_step,
            "l2": "inputs larger than L2 (no flush needed)" if input_bytes > 2 * 129e6
            else "L2 flushed before every step (256 MB write, then a 256 MB read so that the write's dirty "
                 "lines are written back before the step; outside the timed events)",
            "parallelism": parallelism}


class Workload:
    """Device-resident inputs and outputs of one workload, and its step."""

    def __init__(self, name: str, seed_offset: int = 0):
        import gapped_varlen_attention_gb300 as gva
        from gapped_varlen_attention_gb300 import workloads as W
        self.name = name
        self.gva = gva
        dev = "cuda"
        sp = self.spec = spec(name)
        self.label, self.geoms, self.parts = sp.label, sp.geoms, sp.parts
        if sp.ranges is not None:
            self.ranges = sp.ranges
        if sp.causal_block:
            self.causal_block = sp.causal_block
        if sp.backward:
            self.backward = True
        if sp.merge_only:
            self.merge_only = True
            self.used_k_parts = sp.used_k_parts
        elif sp.part_kv_geoms is not None:
            self.q = W.make_qkv(sp.qkv_geom, sp.seed + seed_offset, device=dev)[0]
            self.part_kv = [W.make_qkv(pg, s + seed_offset, device=dev)[1:] for pg, s in sp.part_kv_geoms]
        else:
            self.q, self.k, self.v = W.make_qkv(sp.qkv_geom, sp.seed + seed_offset, device=dev,
                                                k_pad_fill=sp.k_pad_fill)
        self.merge_only = getattr(self, "merge_only", False)
        if self.merge_only:
            self.plans = []
        elif getattr(self, "ranges", None) is not None:
            g = self.geoms[0]
            self.plans = [gva.Plan.from_ranges(g.cu_q, g.used_q, self.ranges, g.total_k, g.num_heads_q,
                                               g.num_heads_kv, g.head_dim)]
        else:
            self.plans = [gva.Plan.from_geometry(g, getattr(self, "causal_block", 0)) for g in self.geoms]
        g0 = self.geoms[0]
        if self.merge_only:
            self.merge_plan = gva.Plan.from_geometry(self.parts)
            self.out, self.lse = W.make_outputs(self.parts, 0.0, device=dev)
            outs, lses = W.make_partials(self.parts, self.used_k_parts, 3004 + seed_offset, device=dev)
            self.partials = list(zip(outs, lses))
        elif self.parts is None:
            self.out, self.lse = W.make_outputs(g0, 0.0, device=dev)
            self.partials = None
        else:
            self.merge_plan = gva.Plan.from_geometry(self.parts)
            self.out, self.lse = W.make_outputs(self.parts, 0.0, device=dev)
            self.partials = [W.make_outputs(p, 0.0, device=dev, out_dtype=torch.float32) for p in self.geoms]
        self.flops = float(sum(p.info()["used_flops"] for p in self.plans))
        self.launches_per_step = len(self.geoms) + (0 if self.parts is None else 1)
        self.metric, self.unit, self.scale, self.bound = METRIC, UNIT, 1e12, "tensor"
        self.kernel = self.kernel_key = "gva_fwd_kernel"
        # the forward launch that dominates the step (most FLOPs)
        self.dominant = int(np.argmax([p.info()["used_flops"] for p in self.plans])) if self.plans else 0
        if getattr(self, "part_kv", None) is not None:
            self.inputs = [self.q] + [t for kv in self.part_kv for t in kv]
        elif not self.merge_only:
            self.inputs = [self.q, self.k, self.v]
        self.outputs = [self.out, self.lse]
        if self.merge_only:
            self.inputs = [t for o_l in self.partials for t in o_l]
            self.launches_per_step = 1
            self.flops = 0.0
            self.metric = "gapped-varlen FP32 LSE merge GB/s (algorithmic bytes: live partials, LSEs, output)"
            self.unit, self.scale, self.bound = "GB/s", 1e9, "hbm"
            self.kernel = "gva_lse_merge_kernel<float, bf16>"
            self.kernel_key = "gva_lse_merge_kernel"
        if getattr(self, "backward", False):
            # the forward's O and LSE are inputs of the backward (computed once, untimed)
            gva.forward(self.plans[0], self.q, self.k, self.v, self.out, self.lse)
            gen = torch.Generator(device=dev).manual_seed(2005 + seed_offset)
            self.d_out = torch.randn(self.q.shape, generator=gen, device=dev).bfloat16()
            self.grads = [torch.empty_like(self.q), torch.empty_like(self.k), torch.empty_like(self.v)]
            self.ws = torch.empty(max(16, gva.backward_workspace_bytes(self.plans[0])), dtype=torch.uint8,
                                  device=dev)
            self.flops *= 2.5
            self.launches_per_step = 3  # rowsum(dO * O), dQ, dK / dV
            self.metric = "gapped-varlen attn bwd TFLOP/s (used rows, 2.5 x fwd FLOPs) & % of GB300 BF16 peak"
            self.kernel = "gva_backward (3 launches: rowsum, dQ, dK/dV)"
            self.kernel_key = "gva_backward"
            self.inputs = [self.q, self.k, self.v, self.out, self.lse, self.d_out]
            self.outputs = list(self.grads)
        self.work = merge_bytes(self.parts, self.used_k_parts, self.out.element_size()) if self.merge_only \
            else self.flops  # the metric's numerator per step (FLOPs, or bytes for the merge)

    def step(self, inputs=None, outputs=None):
        """One pass of the path on the current stream: `inputs` / `outputs` default to the
        workload's resident tensors (same order as self.inputs / self.outputs)."""
        gva = self.gva
        inputs = inputs or self.inputs
        outputs = outputs or self.outputs
        if self.merge_only:
            n = len(self.partials)
            gva.lse_merge(self.merge_plan, inputs[0:2 * n:2], inputs[1:2 * n:2], *outputs)
            return
        q, k, v = inputs[:3]
        if getattr(self, "backward", False):
            out, lse, d_out = inputs[3:]
            gva.backward(self.plans[0], q, k, v, out, lse, d_out, *outputs, workspace=self.ws)
        elif self.partials is None:
            gva.forward(self.plans[0], q, k, v, *outputs)
        else:
            for i, (plan, (o, l)) in enumerate(zip(self.plans, self.partials)):
                ki, vi = self.kv_of(i, inputs)
                gva.forward(plan, q, ki, vi, o, l)
            gva.lse_merge(self.merge_plan, [p[0] for p in self.partials], [p[1] for p in self.partials],
                          *outputs)

    def kv_of(self, i, inputs=None):
        """K and V of forward launch i (each partition has its own buffers, or all share one)."""
        inputs = inputs or self.inputs
        if getattr(self, "part_kv", None) is not None:
            return inputs[1 + 2 * i], inputs[2 + 2 * i]
        return inputs[1], inputs[2]

    def dominant_bytes(self) -> float:
        """Algorithmic HBM bytes of one launch of the dominant kernel (one backward call
        for the backward): each used row and used key read or written once. Forward: Q,
        O and the LSE of the used rows, K and V of the used keys. Backward: Q, O, dO and
        dQ of the used rows, K, V, dK and dV of the used keys, the LSE read and D
        written once and read twice. Merge: the metric's own bytes."""
        if self.merge_only:
            return float(self.work)
        g = self.geoms[0 if getattr(self, "backward", False) else self.dominant]
        hq, hkv, d = g.num_heads_q, g.num_heads_kv, g.head_dim
        q_rows = float(np.sum(g.used_q))
        if getattr(self, "ranges", None) is not None:
            k_rows = float(sum(n for rs in self.ranges for _, n in rs))
        else:
            k_rows = float(np.sum(g.used_k))
        if getattr(self, "backward", False):
            return q_rows * hq * (4 * d * 2 + 4 * 4) + k_rows * hkv * 4 * d * 2
        out = self.partials[self.dominant][0] if self.partials else self.out
        return q_rows * hq * (d * 2 + d * out.element_size() + 4) + k_rows * hkv * 2 * d * 2

    def check(self):
        for p in self.plans + ([self.merge_plan] if self.parts is not None else []):
            self.gva.device_status(p)

    def config(self, parallelism: str):
        per_step = {"algorithmic_bytes_per_step": self.work} if self.merge_only else \
            {"useful_flops_per_step": self.flops}
        return spec_config(self.spec, per_step, parallelism)

    def input_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.inputs)

    def output_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.outputs)

    def row_ranges(self):
        """(inputs, outputs): per tensor, the row ranges along dim 0 that hold data (the
        used rows of every segment), or None for a tensor that is copied whole (LSE and
        D, laid out [heads, rows]). Gap rows are neither inputs nor results."""
        def used(cu, n):
            out = []
            for b in range(len(n)):
                r0, k = int(cu[b]), int(n[b])
                if k == 0:
                    continue
                if out and out[-1][0] + out[-1][1] == r0:
                    out[-1] = (out[-1][0], out[-1][1] + k)
                else:
                    out.append((r0, k))
            return out
        qg = self.parts if self.parts is not None else self.geoms[0]
        q = used(qg.cu_q, qg.used_q)
        if self.merge_only:
            return [q, None] * len(self.partials), [q, None]
        if getattr(self, "part_kv", None) is not None:
            ks = [used(g.cu_k, g.used_k) for g in self.geoms]
            return [q] + [r for k in ks for r in (k, k)], [q, None]
        kg = self.parts if self.parts is not None else self.geoms[0]
        if getattr(self, "ranges", None) is not None:
            k = sorted((st, n) for rs in self.ranges for st, n in rs if n > 0)
        else:
            k = used(kg.cu_k, kg.used_k)
        if getattr(self, "backward", False):
            return [q, k, k, q, None, q], [q, k, k]
        return [q, k, k], [q, None]

    def copy_bytes(self):
        """Bytes the end-to-end steps copy in and out per step (the row ranges above)."""
        def nbytes(ts, rs):
            tot = 0
            for t, r in zip(ts, rs):
                row = t[0].numel() * t.element_size() if t.shape[0] else 0
                tot += t.numel() * t.element_size() if r is None else sum(n for _, n in r) * row
            return tot
        ri, ro = self.row_ranges()
        return nbytes(self.inputs, ri), nbytes(self.outputs, ro)


def merge_bytes(g, used_k_parts, out_bytes: int, rows=None) -> float:
    """Algorithmic bytes of one FP32 LSE merge over g's used rows (or the listed rows):
    every partition's LSE read and the merged LSE written (4 bytes each per row and
    head), each live partition's FP32 output read (a keyless one, LSE = -inf, is
    skipped), and the merged output written."""
    hq, d = g.num_heads_q, g.head_dim
    total = 0.0
    for b in range(g.num_segments):
        n = int(g.used_q[b]) if rows is None else int(np.sum(
            (np.asarray(rows) >= int(g.cu_q[b])) & (np.asarray(rows) < int(g.cu_q[b]) + int(g.used_q[b]))))
        live = sum(1 for uk in used_k_parts if int(uk[b]) > 0)
        total += n * hq * (4.0 * (len(used_k_parts) + 1) + d * (4.0 * live + out_bytes))
    return total


# --------------------------------------------------------------------------------------
# Measurement helpers
# --------------------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_only(text: str) -> str:
    """C / C++ / CUDA source without its comments, blank lines and trailing spaces
    (string and character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash(kernel: str) -> str:
    """sha256[:16] over the code of the kernel's sources (its .cu file, then the headers
    it includes), comments left out: a comment edit leaves a recorded capture valid."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch of the workload's dominant kernel (per call
    for the backward's three launches), from the ncu record, if it was measured on the
    current kernel sources; else None."""
    if not os.path.exists(TRAFFIC_RECORD):
        return None
    with open(TRAFFIC_RECORD) as f:
        rec = json.load(f).get("records", {}).get(workload)
    if not rec or rec.get("kernel") != kernel or rec.get("source_sha16") != kernel_source_hash(kernel):
        return None
    return float(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_samples(self, n: int, timeout_s: float, work=None) -> None:
        """Wait until `n` samples have arrived (at most `timeout_s`), calling `work`
        meanwhile if given (to keep the GPU under the same load)."""
        if self.proc is None:
            return
        t_end = time.monotonic() + timeout_s
        while len(self.lines) < n and time.monotonic() < t_end:
            if work is None:
                time.sleep(0.02)
            else:
                work()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


class L2Flush:
    """Leaves L2 cold before a timed step: writes a 256 MB buffer (twice the 129 MB L2),
    then reads another 256 MB, so that L2 holds only clean lines of neither input nor
    output and the write-back of the written lines is not charged to the step."""

    def __init__(self):
        self.dirty = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.clean = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
        self.acc = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self):
        self.dirty.fill_(1)
        torch.sum(self.clean, dim=0, out=self.acc)


def time_steps(fn, steps: int, stream, flush=None, per_step=None) -> float:
    """Device milliseconds for `steps` calls of fn, CUDA events on `stream`. With a
    flush (an L2Flush, for inputs smaller than L2), it runs before every step, outside
    the events, so each step starts with a cold L2 and only the step is timed; a short
    device-side sleep after it covers the host's time to issue the step. Without one the
    steps run back to back, with an event between consecutive steps. `per_step`, if
    given, receives each step's milliseconds."""
    if flush is None:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        ev[0].record(stream)
        for i in range(steps):
            fn()
            ev[i + 1].record(stream)
        ev[-1].synchronize()
        if per_step is not None:
            per_step.extend(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))
        return ev[0].elapsed_time(ev[-1])
    pairs = []
    for _ in range(steps):
        flush()
        # keep the device busy (outside the events) while the host issues the step, so
        # that a short step is timed from its first launch, not from the host's call
        torch.cuda._sleep(200000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        pairs.append((a, b))
    pairs[-1][1].synchronize()
    if per_step is not None:
        per_step.extend(a.elapsed_time(b) for a, b in pairs)
    return sum(a.elapsed_time(b) for a, b in pairs)


def copy_rows(dst, src, ranges):
    """Asynchronous copy of the listed row ranges (dim 0), or of the whole tensor."""
    if ranges is None:
        dst.copy_(src, non_blocking=True)
        return
    for r0, n in ranges:
        dst[r0:r0 + n].copy_(src[r0:r0 + n], non_blocking=True)


class E2EPipeline:
    """Steps through the public API with host buffers: for every step, the host->device
    copy of its inputs (pinned host memory), the step, and the device->host copy of its
    results. Two device buffer sets and two copy streams let step i+1's input copy and
    step i-1's result copy run while step i computes; each step still makes all of its
    own copies, and the timed region ends when the last result is on the host."""

    def __init__(self, wl, stream):
        self.wl, self.stream = wl, stream
        self.r_in, self.r_out = wl.row_ranges()
        self.h_in = [t.cpu().pin_memory() for t in wl.inputs]
        self.d_in = [[torch.empty_like(t) for t in wl.inputs] for _ in range(2)]
        self.d_out = [[torch.empty_like(t) for t in wl.outputs] for _ in range(2)]
        self.h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in wl.outputs] for _ in range(2)]
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def run(self, steps: int) -> float:
        """Device milliseconds for `steps` end-to-end steps. `self.compute_ms` receives
        each step's own time on the compute stream (from the end of its waits for its
        input copy and its buffers to the end of the step), so that the region's time
        splits into compute under concurrent copies and what the copies add."""
        st = self.stream
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        bracket = []
        start.record(st)
        self.s_in.wait_stream(st)
        self.s_out.wait_stream(st)
        computed = [None, None]  # per buffer set: the step that last read it has finished
        copied = [None, None]    # per buffer set: its results are on the host
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(self.s_in):
                if computed[b] is not None:
                    self.s_in.wait_event(computed[b])
                for d, h, r in zip(self.d_in[b], self.h_in, self.r_in):
                    copy_rows(d, h, r)
                loaded = torch.cuda.Event()
                loaded.record(self.s_in)
            st.wait_event(loaded)
            if copied[b] is not None:
                st.wait_event(copied[b])
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            self.wl.step(self.d_in[b], self.d_out[b])
            z.record(st)
            bracket.append((a, z))
            computed[b] = torch.cuda.Event()
            computed[b].record(st)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(computed[b])
                for h, d, r in zip(self.h_out[b], self.d_out[b], self.r_out):
                    copy_rows(h, d, r)
                copied[b] = torch.cuda.Event()
                copied[b].record(self.s_out)
        st.wait_stream(self.s_in)
        st.wait_stream(self.s_out)
        end.record(st)
        end.synchronize()
        self.compute_ms = [a.elapsed_time(z) for a, z in bracket]
        return start.elapsed_time(end)

    def copy_rates(self, reps: int = 3):
        """GB/s of one step's own copies run alone, nothing else on the device: the
        host->device copy of its inputs and the device->host copy of its results (the
        same row ranges and pinned buffers as the timed steps), each timed with events
        on its copy stream. They tell how much of an end-to-end step the box's copy
        rate sets."""
        rates = []
        for stream, copies in ((self.s_in, [(d, h, r) for d, h, r in zip(self.d_in[0], self.h_in, self.r_in)]),
                               (self.s_out, [(h, d, r) for h, d, r in zip(self.h_out[0], self.d_out[0],
                                                                          self.r_out)])):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                for _ in range(reps):
                    for dst, src, r in copies:
                        copy_rows(dst, src, r)
                b.record(stream)
            b.synchronize()
            rates.append(a.elapsed_time(b) / reps)
        bi, bo = self.wl.copy_bytes()
        return {"h2d_gbs": round(bi / (rates[0] * 1e-3) / 1e9, 1) if rates[0] > 0 else None,
                "d2h_gbs": round(bo / (rates[1] * 1e-3) / 1e9, 1) if rates[1] > 0 else None,
                "h2d_ms": round(rates[0], 4), "d2h_ms": round(rates[1], 4)}


def max_over_ranks(values, dist, device):
    """Element-wise maximum of per-rank timings over all ranks (the slowest rank sets
    the job's time); the identity without a process group."""
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rate(world: int, work_per_rank: float, ms: float, scale: float = 1e12) -> float:
    """Whole-job throughput: every rank runs its own copy of the workload (weak scaling),
    so the job does world x the per-rank work (FLOPs or bytes) in the slowest rank's
    time; ``scale`` 1e12 gives TFLOP/s, 1e9 GB/s."""
    return world * work_per_rank / (ms * 1e-3) / scale


def job_tflops(world: int, flops_per_rank: float, ms: float) -> float:
    return job_rate(world, flops_per_rank, ms, 1e12)


# --------------------------------------------------------------------------------------
# CPU oracle timing (the reported baseline)
# --------------------------------------------------------------------------------------

def oracle_sample_rate(wl, budget_s: float, seed: int = 0):
    """Run the FP64 oracle on a seeded sample of used rows of the workload for about
    `budget_s` seconds; return (TFLOP/s, description, rows, seconds)."""
    from oracle import gva_oracle
    geoms = wl.geoms
    rng = np.random.default_rng(seed)
    if getattr(wl, "merge_only", False):
        return oracle_merge_rate(wl, budget_s, rng)
    q = wl.q.cpu()
    part_kv = getattr(wl, "part_kv", None)
    if part_kv is not None:
        kvs = [(k_.cpu(), v_.cpu()) for k_, v_ in part_kv]
    else:
        kvs = [(wl.k.cpu(), wl.v.cpu())] * len(geoms)
    backward = getattr(wl, "backward", False)
    cb = getattr(wl, "causal_block", 0)
    d_out = wl.d_out.cpu() if backward else None
    done_flops = 0.0
    rows_done = 0
    t0 = time.perf_counter()
    while True:
        for g, (k, v) in zip(geoms, kvs):
            b = int(rng.choice(np.flatnonzero(g.used_q > 0)))
            local = [int(x) for x in rng.integers(0, int(g.used_q[b]), size=4)]
            rows = [int(g.cu_q[b]) + r for r in local]
            k0, nk = int(g.cu_k[b]), int(g.used_k[b])
            # keys each sampled row sees (all used keys, or its block-causal prefix)
            vis = (gva_oracle.causal_limits(int(g.used_q[b]), nk, cb)[local] if cb > 0
                   else np.full(len(local), nk))
            if backward and cb == 0:
                # the sampled rows as one segment over their segment's keys: all five products
                gva_oracle.attention_backward(q[rows], k[k0:k0 + nk], v[k0:k0 + nk], d_out[rows], [0, len(rows)],
                                              [len(rows)], [0, nk], [nk])
                done_flops += 10.0 * g.head_dim * g.num_heads_q * float(np.sum(vis))
            elif backward:
                # block-causal: each sampled row as its own segment over the keys it sees
                for r, n in zip(rows, vis):
                    gva_oracle.attention_backward(q[[r]], k[k0:k0 + int(n)], v[k0:k0 + int(n)], d_out[[r]],
                                                  [0, 1], [1], [0, int(n)], [int(n)])
                done_flops += 10.0 * g.head_dim * g.num_heads_q * float(np.sum(vis))
            else:
                gva_oracle.attention_rows(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k, rows, causal_block=cb)
                done_flops += 4.0 * g.head_dim * g.num_heads_q * float(np.sum(vis))
            rows_done += len(rows)
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    what = "backward of " if backward else ""
    keys = "every key each row sees" if cb > 0 else "every used key of their segment"
    desc = (f"{what}{rows_done} seeded used rows (all {geoms[0].num_heads_q} heads, {keys}) of the {wl.name} "
            f"workload, FP64 NumPy oracle")
    return done_flops / el / 1e12, desc, rows_done, el


def oracle_merge_rate(wl, budget_s: float, rng):
    """The FP64 oracle merge on seeded samples of 64 used rows of the merge workload for
    about `budget_s` seconds; return (GB/s of algorithmic bytes, description, rows, seconds)."""
    from oracle import gva_oracle
    g = wl.parts
    outs = [o.cpu().numpy() for o, _ in wl.partials]
    lses = [l_.cpu().numpy() for _, l_ in wl.partials]
    used_rows = np.concatenate([np.arange(int(g.cu_q[b]), int(g.cu_q[b]) + int(g.used_q[b]))
                                for b in range(g.num_segments)])
    done, rows_done = 0.0, 0
    t0 = time.perf_counter()
    while True:
        rows = np.sort(rng.choice(used_rows, size=64, replace=False))
        gva_oracle.lse_merge([o[rows] for o in outs], [x[:, rows] for x in lses], [0, len(rows)], [len(rows)])
        done += merge_bytes(g, wl.used_k_parts, 2, rows=rows)
        rows_done += len(rows)
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    desc = (f"{rows_done} seeded used rows (all {g.num_heads_q} heads, {len(outs)} FP32 partitions) of the "
            f"{wl.name} workload, FP64 NumPy oracle merge")
    return done / el / 1e9, desc, rows_done, el


# --------------------------------------------------------------------------------------

# the other workloads the default run also measures (one entry each in `configs`):
# the pages' remaining shapes, the fused and block-causal forms of the multiview replay,
# the merge alone and the backward of the long replay
CONFIG_WORKLOADS = ("tiny", "cfg_text_cross", "multiview_causal", "multiview_fused", "multiview_blockcausal",
                    "lse_merge_union", "lse_merge", "long_replay_bwd")


def measure(wl, steps: int, warmup: int, e2e_steps: int, stream, clock_index: int, barrier=lambda: None):
    """Time one workload on this rank: `steps` steps (CUDA events per step), the
    dominant kernel alone, the end-to-end steps through the public API, the pinned copy
    rates, and the SM clocks during the timed region. Returns the raw numbers."""
    for _ in range(warmup):
        wl.step()
    torch.cuda.synchronize()
    wl.check()
    flush = L2Flush() if spec_input_bytes(wl.spec) <= 2 * 129e6 else None
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(clock_index) as clocks:
        # nvidia-smi is up before the timed region starts; the same steps keep running
        # meanwhile so that the clocks do not drop while the device would otherwise idle
        def keep_busy():
            for _ in range(max(1, warmup)):
                wl.step()
            torch.cuda.synchronize()
        clocks.wait_samples(1, 5.0, work=keep_busy)
        n_before = len(clocks.lines)
        torch.cuda.nvtx.range_push("timed")  # lets a profiler keep only the timed launches
        step_ms = []
        ms = time_steps(wl.step, steps, stream, flush, step_ms)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        window = "timed region"
        if len(clocks.lines) - n_before < 3:
            # a timed region shorter than the 200 ms sampling period: sample the same
            # steps, untimed, right after it
            def more():
                for _ in range(4):
                    wl.step()
                torch.cuda.synchronize()
            clocks.wait_samples(n_before + 3, 3.0, work=more)
            window = ("timed region plus the same steps, untimed, right after it (the region is shorter than "
                      "the sampling period)")
    barrier()
    # kernel-only time of the dominant launch (the forward with the most FLOPs; for the
    # backward workload the whole backward call, for the merge workload the merge)
    if getattr(wl, "backward", False) or wl.merge_only:
        dominant = wl.step
    else:
        i = wl.dominant
        dominant = lambda: wl.gva.forward(wl.plans[i], wl.q, *wl.kv_of(i),  # noqa: E731
                                          *(wl.partials[i] if wl.partials else (wl.out, wl.lse)))
    n_dom = max(3, steps // 2)
    dom_ms = time_steps(dominant, n_dom, stream, flush) / n_dom
    wl.check()
    same_size_copy_gbs = None
    if wl.bound == "hbm":
        # context for an HBM-bound kernel of this size: a device copy moving the same
        # bytes (half read, half written), timed the same way
        src = torch.empty(int(wl.work // 2), dtype=torch.uint8, device="cuda")
        dst = torch.empty_like(src)
        copy_ms = time_steps(lambda: dst.copy_(src), 10, stream, flush) / 10
        same_size_copy_gbs = wl.work / (copy_ms * 1e-3) / 1e9
        del src, dst
    # end to end through the public API: every step copies its inputs from pinned host
    # memory and its results back, inside the timed region (pipelined over two buffers)
    e2e_run = E2EPipeline(wl, stream)
    e2e_run.run(1)
    torch.cuda.synchronize()
    barrier()
    with ClockSampler(clock_index) as e2e_clocks:
        e2e_clocks.wait_samples(1, 5.0, work=lambda: (e2e_run.run(1), torch.cuda.synchronize()))
        e2e_ms = e2e_run.run(e2e_steps) / e2e_steps
    e2e_compute_ms = float(np.mean(e2e_run.compute_ms))
    barrier()
    copy = e2e_run.copy_rates()
    del e2e_run
    return {"ms_step": ms / steps, "med_ms": float(np.median(step_ms)), "dom_ms": dom_ms, "dom_launches": n_dom,
            "e2e_ms": e2e_ms, "e2e_steps": e2e_steps, "e2e_compute_ms": e2e_compute_ms,
            "e2e_clocks": e2e_clocks.summary(),
            "copy": copy, "clocks": {**clocks.summary(), "window": window},
            "same_size_copy_gbs": same_size_copy_gbs, "l2_flushed": flush is not None}


def roofline_of(wl, r, peaks, peak_src, traffic):
    """The roofline entry of the dominant kernel. Its peak is the measured burst rate
    when the kernel's own timed region (dom_launches x dom_ms) lasts under a second,
    else the sustained one; both fractions are given for tensor-bound kernels."""
    if getattr(wl, "backward", False) or wl.merge_only:
        dom_work = wl.work
    else:
        dom_work = wl.plans[wl.dominant].info()["used_flops"]
    achieved = dom_work / (r["dom_ms"] * 1e-3) / wl.scale
    region_ms = r["dom_ms"] * r["dom_launches"]
    out = {"bound": wl.bound, "achieved": round(achieved, 2)}
    if wl.bound == "hbm":
        peak = peaks["hbm_gbs"]
        out.update(peak=peak, unit=wl.unit, frac=round(achieved / peak, 4),
                   peak_source=f"{peak_src} HBM copy bandwidth (STREAM-style, read + write bytes)")
    else:
        sustained = region_ms > 1000.0
        peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        out.update(peak=peak, unit=wl.unit, frac=round(achieved / peak, 4),
                   frac_burst=round(achieved / peaks["bf16_tflops"], 4),
                   frac_sustained=round(achieved / peaks["bf16_tflops_sustained"], 4),
                   peak_source=(f"{peak_src} {'sustained' if sustained else 'burst'} dense bf16 (cuBLAS): the "
                                f"kernel's timed region ({r['dom_launches']} launches, {region_ms:.0f} ms) is "
                                f"{'over' if sustained else 'under'} 1 s"))
    out.update(traffic=traffic, kernel=wl.kernel, ms_per_launch=round(r["dom_ms"], 4),
               launches_timed=r["dom_launches"])
    alg = wl.dominant_bytes()
    out["algorithmic_bytes"] = alg
    if traffic is not None and alg > 0:
        out["traffic_over_algorithmic"] = round(traffic / alg, 3)
    if r["same_size_copy_gbs"] is not None:
        out["same_size_copy_gbs"] = round(r["same_size_copy_gbs"], 1)
    return out


def e2e_of(wl, r, world):
    bi, bo = wl.copy_bytes()
    return {"value": round(job_rate(world, wl.work, r["e2e_ms"], wl.scale), 3), "unit": wl.unit,
            "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo), "ms_per_step": round(r["e2e_ms"], 4),
            "copy_gbs": r["copy"],
            "steps": r["e2e_steps"],
            "compute_ms_per_step": round(r["e2e_compute_ms"], 4),
            "resident_ms_per_step": round(r["ms_step"], 4),
            "clocks": r["e2e_clocks"],
            "copies": "pinned host buffers; every step copies its inputs in and its results out: the used rows of "
                      "each [rows, heads, d] tensor (gap rows are neither inputs nor results) and whole LSE-shaped "
                      "tensors; two device buffer sets and two copy streams overlap step i+1's input copy and step "
                      "i-1's result copy with step i. copy_gbs: the same copies run alone on this box. "
                      "compute_ms_per_step: each step's own time on the compute stream inside this region (the "
                      "copies of other steps running beside it), against resident_ms_per_step, the same step "
                      "with no copies; the first step's input copy and the last step's result copy have no step to "
                      "hide behind, so they add (h2d_ms + d2h_ms) / steps per step; clocks: sampled during this region"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gva", "reference"], default="gva")
    ap.add_argument("--workload", default="long_replay", choices=list(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--configs", default="auto",
                    help="comma-separated workloads measured after the main one and reported under `configs`; "
                         "'auto': the other workloads for the default run, none otherwise; 'none': none")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3 and args.impl == "gva":
        args.warmup = 3

    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    import gapped_varlen_attention_gb300 as gva
    if rank == 0 or world == 1:
        gva.build()
    if dist is not None:
        dist.barrier()
    gva.load_library()
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()

    if args.configs == "auto":
        extra = [w for w in CONFIG_WORKLOADS if w != args.workload] if args.workload == "long_replay" else []
    elif args.configs == "none":
        extra = []
    else:
        extra = [w for w in args.configs.split(",") if w and w != args.workload]
        for w in extra:
            if w not in LABELS:
                raise SystemExit(f"unknown workload {w}")

    wl = Workload(args.workload, seed_offset=rank)
    r = measure(wl, args.steps, args.warmup, args.e2e_steps, stream, local_rank, barrier)
    r["ms_step"], r["dom_ms"], r["e2e_ms"], r["med_ms"] = max_over_ranks(
        [r["ms_step"], r["dom_ms"], r["e2e_ms"], r["med_ms"]], dist, "cuda")
    peaks, peak_src = load_peaks()
    cpu = oracle_sample_rate(wl, args.cpu_budget_s) if rank == 0 else None

    configs = {}
    for name in extra:
        # the main workload's buffers stay resident; each extra workload is built, timed
        # and released in turn
        w = Workload(name, seed_offset=rank)
        rc = measure(w, args.steps, args.warmup, args.e2e_steps, stream, local_rank, barrier)
        rc["ms_step"], rc["dom_ms"], rc["e2e_ms"], rc["med_ms"] = max_over_ranks(
            [rc["ms_step"], rc["dom_ms"], rc["e2e_ms"], rc["med_ms"]], dist, "cuda")
        value = job_rate(world, w.work, rc["ms_step"], w.scale)
        configs[name] = {
            "description": w.label, "metric": w.metric, "unit": w.unit,
            "value": round(value, 3), "ms_per_step": round(rc["ms_step"], 4),
            "ms_per_step_median": round(rc["med_ms"], 4),
            ("algorithmic_bytes_per_step" if w.merge_only else "useful_flops_per_step"): w.work,
            "roofline": roofline_of(w, rc, peaks, peak_src, recorded_traffic(name, w.kernel_key)),
            "e2e": e2e_of(w, rc, world),
            "gpu_launches": args.steps * w.launches_per_step,
            "clocks": rc["clocks"],
            "l2": "flushed before every step" if rc["l2_flushed"] else "inputs larger than L2",
        }
        del w
        torch.cuda.empty_cache()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    value = job_rate(world, wl.work, r["ms_step"], wl.scale)
    peak_line = peaks["hbm_gbs"] if wl.bound == "hbm" else peaks[
        "bf16_tflops_sustained" if args.steps * r["ms_step"] > 1000.0 else "bf16_tflops"]
    cpu_rate, cpu_desc, _, _ = cpu
    line = {
        "metric": wl.metric,
        "value": round(value, 3),
        "unit": wl.unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(r["ms_step"], 4),
        "ms_per_step_median": round(r["med_ms"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, the pages' segment shapes)",
        "config": wl.config(f"replicas x{world} (independent problems per GPU)"),
        ("pct_of_hbm_peak" if wl.bound == "hbm" else "pct_of_bf16_peak"): round(
            100.0 * value / world / peak_line, 2),
        **({} if wl.bound == "hbm" else {
            "pct_of_bf16_peak_burst": round(100.0 * value / world / peaks["bf16_tflops"], 2),
            "pct_of_bf16_peak_sustained": round(100.0 * value / world / peaks["bf16_tflops_sustained"], 2)}),
        "roofline": roofline_of(wl, r, peaks, peak_src, recorded_traffic(args.workload, wl.kernel_key)),
        "e2e": e2e_of(wl, r, world),
        "gpu_launches": args.steps * wl.launches_per_step,
        "clocks": r["clocks"],
        "cpu_baseline": {"value": round(cpu_rate, 6), "unit": wl.unit, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": cpu_desc},
    }
    if configs:
        line["configs"] = configs
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args, world, rank):
    """The oracle, timed as it stands on the host cores, on bounded samples of the same
    workload: each step is a seeded sample of used rows sized to ~budget seconds."""
    if rank != 0:
        return
    from gapped_varlen_attention_gb300 import workloads as W
    from oracle import gva_oracle

    sp = spec(args.workload)
    wl = types.SimpleNamespace(name=sp.name, geoms=sp.geoms, causal_block=sp.causal_block, backward=sp.backward)
    metric, unit = METRIC, UNIT
    if sp.merge_only:
        wl.merge_only, wl.parts, wl.used_k_parts = True, sp.parts, sp.used_k_parts
        wl.partials = list(zip(*W.make_partials(sp.parts, sp.used_k_parts, 3004)))
        metric, unit = "gapped-varlen FP32 LSE merge GB/s (algorithmic bytes: live partials, LSEs, output)", "GB/s"
        per_step = {"algorithmic_bytes_per_step": merge_bytes(sp.parts, sp.used_k_parts, 2)}
    else:
        if sp.part_kv_geoms is not None:
            wl.q = W.make_qkv(sp.qkv_geom, sp.seed)[0]
            wl.part_kv = [W.make_qkv(pg, s)[1:] for pg, s in sp.part_kv_geoms]
        else:
            wl.q, wl.k, wl.v = W.make_qkv(sp.qkv_geom, sp.seed, k_pad_fill=sp.k_pad_fill)
        # the workload's useful FLOPs, counted on the host: used (or visible) pairs x 4 d Hq
        flops = 0.0
        for g in sp.geoms:
            if sp.causal_block:
                pairs = sum(float(gva_oracle.causal_limits(int(g.used_q[b]), int(g.used_k[b]), sp.causal_block).sum())
                            for b in range(g.num_segments))
                flops += 4.0 * g.head_dim * g.num_heads_q * pairs
            else:
                flops += gva_oracle.used_flops(g.used_q, g.used_k, g.num_heads_q, g.head_dim)
        if sp.backward:
            wl.d_out = torch.randn(wl.q.shape, generator=torch.Generator().manual_seed(2005)).bfloat16()
            metric = "gapped-varlen attn bwd TFLOP/s (used rows, 2.5 x fwd FLOPs) & % of GB300 BF16 peak"
            flops *= 2.5
        per_step = {"useful_flops_per_step": flops}
    config = spec_config(sp, per_step, "FP64 oracle on the host cores (rank 0 only)")
    budget = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_sample_rate(wl, budget, seed=i)
    rates, descs, secs = [], [], 0.0
    for i in range(args.steps):
        r, d, _, el = oracle_sample_rate(wl, budget, seed=100 + i)
        rates.append(r)
        descs.append(d)
        secs += el
    value = float(np.mean(rates))
    line = {
        "impl": "reference",
        "metric": metric,
        "value": round(value, 6),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 widened to f64)",
        "config": config,
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": descs[-1] + f"; {budget:.1f} s per step"},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
