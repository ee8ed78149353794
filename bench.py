"""Benchmark of the block-quantized decode matvec on GB300.

One step = one pass over every hot-path row of the method, each on its own
weights resident in HBM:
  * NVFP4 GEMV, N = 1: 12288x4096, 4096x12288, 4096x4096 (ts = 0.01)
  * Q8_0 GEMV, N = 1: 12288x4096, 4096x12288, 151936x4096 (LM head)
  * speculative verify, NVFP4, N = 4 and 8: 4096x4096, 12288x4096
  * routed MoE layer (256 experts, H 2048, I 512, top-8): T = 1 and T = 16
    (router + expert-major list + grouped gate_up/SiLU*up + grouped down +
    combine)
The metric is algorithmic HBM bytes (packed weights + scales + activations +
outputs; MoE: the experts the routing actually selects) per second; a step
touches ~1.1 GB, far more than L2, so successive steps read from HBM.

Per row, beside the step: an isolated call after an L2 flush, and calls back
to back (200 graph-captured calls cycling through weight copies whose calls
stream more than 3x L2), each as GB/s and a fraction of the measured HBM
copy peak, with the row's ncu DRAM traffic where a record of the current
kernel sources exists. The 256 x 512 NVFP4 workload is reported the same way
but is not part of the step.

Printed: one JSON line (rank 0). `--impl reference` times the fp64 CPU
oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_quantized_decode_nvfp4_gb300 import synthetic as syn  # noqa: E402

METRIC = "quantized GEMV HBM GB/s & % of GB300 roofline at N=1/4/8; MoE layer us/token"
WORKLOAD = ("decode step: NVFP4 N=1 {12288x4096, 4096x12288, 4096x4096}; Q8_0 N=1 {12288x4096, 4096x12288, "
            "151936x4096}; NVFP4 verify N=4,8 {4096x4096, 12288x4096}; MoE E=256 H=2048 I=512 top-8 T=1,16")
L2_BYTES_FALLBACK = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------- workload
def nvfp4_bytes(M, K, N):
    return M * K // 2 + M * K // 16 + 4 + N * K * 2 + N * M * 4


def q8_0_bytes(M, K, N):
    return M * K + M * (K // 32) * 2 + N * K * 2 + N * M * 4


def moe_expert_bytes(H, I):
    return 2 * I * (H // 2 + H // 16) + H * (I // 2 + I // 16) + 8


def moe_unique_experts(logits, topk):
    sel = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :topk]
    return len(np.unique(sel))


def moe_bytes(T, E, H, I, topk, logits):
    return (moe_unique_experts(logits, topk) * moe_expert_bytes(H, I) + T * H * 2 + T * H * 4 + T * E * 4)


def moe_launches(T, E, H, I, topk):
    """Kernel launches of one moe_layer call: the two batched kernels
    (routing inside them, combine inside the down kernel) for up to 16
    tokens, else route, gate_up, down and combine (plus the status word's
    memset)."""
    small = (T <= 16 and T * topk <= 128 and E <= 512 and H in (1024, 2048, 4096, 8192) and I in (256, 512, 1024)
             and H >= 2 * I and topk * I <= 8192 and T * H <= 32768)
    return 2 if small else 4


def rows_spec():
    """(name, kind, params) of every row of a step, in step order."""
    rows = []
    for M, K in syn.NVFP4_SHAPES:
        rows.append((f"nvfp4 {M}x{K} N=1", "nvfp4", dict(M=M, K=K, N=1)))
    for M, K in syn.Q8_0_SHAPES:
        rows.append((f"q8_0 {M}x{K} N=1", "q8_0", dict(M=M, K=K, N=1)))
    for M, K in syn.VERIFY_SHAPES:
        for N in (4, 8):
            rows.append((f"nvfp4 {M}x{K} N={N}", "nvfp4", dict(M=M, K=K, N=N)))
    for T in (1, 16):
        rows.append((f"moe T={T}", "moe", dict(T=T, E=256, H=2048, I=512, topk=8)))
    return rows


def extra_rows_spec():
    """Rows reported beside the step but not part of it: the tiny 256 x 512
    NVFP4 workload (ts = 1.0), whose time is launch latency, not bandwidth;
    the decode-path epilogue fusions on the layer shapes (gate_up with
    SiLU * up on the 12288 x 4096 gate/up weight, I = 6144; down with the
    residual add on 4096 x 12288); the Q4_0 and FP8 block-128 GEMVs on the
    two layer shapes and the Q4_1 GEMV (CUDA-core path) on 12288 x 4096;
    the tensor-core prefill GEMM of the 12288 x 4096 weight over 2048
    tokens and its grouped form over 256 experts (the MoE gate_up, 2I = 1024
    rows, H = 2048) for 2048 tokens routed top-8 (16384 pairs, multinomial
    expert counts), both reported in TFLOP/s against the measured bf16 peak;
    the whole routed MoE layer for a 1024-token prefill (E = 256, H = 2048,
    I = 512, top-8: routing, gather, both grouped GEMMs, SiLU * up, combine;
    flops 2 * T * topk * 3 * H * I, bytes the experts routed to once, x, y
    and the logits); and the bf16 -> NVFP4 / Q8_0 encoders on a 12288 x 4096
    weight (bytes: bf16 read, codes and scales written)."""
    return [("nvfp4 256x512 N=1", "nvfp4_tiny", dict(M=256, K=512, N=1)),
            ("nvfp4 gate_up+SiLU 12288x4096 N=1", "nvfp4_silu", dict(M=12288, K=4096, N=1)),
            ("nvfp4 down+residual 4096x12288 N=1", "nvfp4_add", dict(M=4096, K=12288, N=1)),
            ("q4_0 12288x4096 N=1", "q4_0", dict(M=12288, K=4096, N=1)),
            ("q4_0 4096x12288 N=1", "q4_0", dict(M=4096, K=12288, N=1)),
            ("q4_1 12288x4096 N=1", "q4_1", dict(M=12288, K=4096, N=1)),
            ("fp8_b128 12288x4096 N=1", "fp8_b128", dict(M=12288, K=4096, N=1)),
            ("fp8_b128 4096x12288 N=1", "fp8_b128", dict(M=4096, K=12288, N=1)),
            ("nvfp4 prefill GEMM 12288x4096 T=2048", "nvfp4_gemm", dict(M=12288, K=4096, N=2048)),
            ("nvfp4 grouped prefill GEMM E=256 1024x2048 P=16384", "nvfp4_gemm_grouped",
             dict(E=256, M=1024, K=2048, N=16384)),
            ("moe prefill T=1024", "moe_prefill", dict(T=1024, E=256, H=2048, I=512, topk=8)),
            ("nvfp4 encode 12288x4096", "nvfp4_encode", dict(M=12288, K=4096, N=1)),
            ("q8_0 encode 12288x4096", "q8_0_encode", dict(M=12288, K=4096, N=1))]


def host_inputs(kind, p, seed=0):
    if kind == "nvfp4_tiny":
        return syn.tiny_nvfp4(seed=seed)
    if kind in ("nvfp4", "nvfp4_silu", "nvfp4_gemm"):
        return syn.dense_nvfp4(p["M"], p["K"], N=p["N"], seed=seed)
    if kind == "nvfp4_gemm_grouped":
        rc, rs, rx, rn = syn.streams(seed, 4)
        E, M, K, P = p["E"], p["M"], p["K"], p["N"]
        w = syn.nvfp4_weight(E * M, K, 0.01, rc, rs)
        counts = rn.multinomial(P, np.ones(E) / E)
        return {"codes": w["codes"], "scales": w["scales"], "ts": np.full(E, 0.01, dtype=np.float32),
                "offsets": np.concatenate([[0], np.cumsum(counts)]).astype(np.int32),
                "x": syn.bf16_normal((P, K), rx)}
    if kind in ("nvfp4_encode", "q8_0_encode"):
        return {"x": syn.bf16_normal((p["M"], p["K"]), np.random.default_rng(seed + 7))}
    if kind == "nvfp4_add":
        h = syn.dense_nvfp4(p["M"], p["K"], N=p["N"], seed=seed)
        h["r"] = np.random.default_rng(seed + 1).standard_normal((p["N"], p["M"])).astype(np.float32)
        return h
    if kind == "q8_0":
        return syn.dense_q8_0(p["M"], p["K"], N=p["N"], seed=seed)
    if kind == "q4_0":
        return syn.dense_q4_0(p["M"], p["K"], N=p["N"], seed=seed)
    if kind == "q4_1":
        return syn.dense_q4_1(p["M"], p["K"], N=p["N"], seed=seed)
    if kind == "fp8_b128":
        return syn.dense_fp8_b128(p["M"], p["K"], N=p["N"], seed=seed)
    return syn.moe_layer(T=p["T"], E=p["E"], H=p["H"], I=p["I"], topk=p["topk"], seed=seed)


def row_bytes(kind, p, host):
    if kind in ("nvfp4", "nvfp4_tiny", "nvfp4_gemm"):
        return nvfp4_bytes(p["M"], p["K"], p["N"])
    if kind == "nvfp4_gemm_grouped":  # every expert's weight once, the tokens, the outputs
        return p["E"] * p["M"] * p["K"] * 9 // 16 + 2 * p["N"] * p["K"] + 4 * p["N"] * p["M"]
    if kind == "nvfp4_silu":  # the output is h, half the rows
        return nvfp4_bytes(p["M"], p["K"], p["N"]) - 4 * p["N"] * p["M"] // 2
    if kind == "nvfp4_add":  # the residual is read
        return nvfp4_bytes(p["M"], p["K"], p["N"]) + 4 * p["N"] * p["M"]
    if kind == "nvfp4_encode":
        return p["M"] * p["K"] * 2 + p["M"] * p["K"] // 2 + p["M"] * p["K"] // 16
    if kind == "q8_0_encode":
        return p["M"] * p["K"] * 2 + p["M"] * p["K"] + p["M"] * p["K"] // 16
    if kind == "q8_0":
        return q8_0_bytes(p["M"], p["K"], p["N"])
    if kind == "q4_0":  # 16 code bytes and a 2-byte scale per 32 weights
        return p["M"] * p["K"] // 2 + p["M"] * (p["K"] // 32) * 2 + 2 * p["N"] * p["K"] + 4 * p["N"] * p["M"]
    if kind == "q4_1":  # 16 code bytes and two 2-byte fields (d, m) per 32 weights
        return p["M"] * p["K"] // 2 + p["M"] * (p["K"] // 32) * 4 + 2 * p["N"] * p["K"] + 4 * p["N"] * p["M"]
    if kind == "fp8_b128":  # a byte per weight, a 4-byte scale per 128 x 128 tile
        return (p["M"] * p["K"] + ((p["M"] + 127) // 128) * ((p["K"] + 127) // 128) * 4 + 2 * p["N"] * p["K"]
                + 4 * p["N"] * p["M"])
    return moe_bytes(p["T"], p["E"], p["H"], p["I"], p["topk"], host["logits"])


# ---------------------------------------------------------------- peaks, clocks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s of a kernel timed alone (the burst figure)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    return FALLBACK_BF16_TFLOPS


class ClockSampler:
    """nvidia-smi clock / throttle samples while running (100 ms period)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [s.strip() for s in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_sha(files=None):
    """Hash of the kernel sources: the named files of csrc/ (a kernel, its
    launcher and the headers they include), or all of csrc/."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantized_decode_nvfp4_gb300", "csrc")
    for f in sorted(files if files else os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(row_key):
    """DRAM bytes per call of a row (all its kernels) from the committed ncu
    record, if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(row_key)
    if not ent or ent.get("source_sha") != source_sha(ent.get("sources")):
        return None
    return ent.get("dram_bytes_per_launch")


def rotating_copies(call_bytes, weight_bytes, l2, mem_budget):
    """Weight copies that a back-to-back loop cycles through so that a call's
    weights are out of L2 when they come round again: the working set of
    the copies' calls must exceed 3x L2 (at least 2 copies, within budget)."""
    r = math.ceil(3 * l2 / max(1, call_bytes)) + 1
    r = min(r, max(2, mem_budget // max(1, weight_bytes)))
    return max(2, r)


# ---------------------------------------------------------------- multi-rank helpers
def max_over_ranks(seconds: float, world: int, device) -> float:
    """The slowest rank's time; every rank calls this (a collective)."""
    if world == 1:
        return seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(step_bytes: int, world: int, steps: int, seconds: float) -> float:
    """Weak scaling: each rank streams step_bytes per step; the job's rate is
    the bytes of all ranks over the slowest rank's time."""
    return step_bytes * world * steps / seconds / 1e9


# ---------------------------------------------------------------- device rows
class Row:
    """One row of the step with its device buffers and launch closure."""

    def __init__(self, name, kind, p, host, torch, bqd):
        self.name, self.kind, self.p = name, kind, p
        self.bytes = row_bytes(kind, p, host)
        self.torch, self.bqd = torch, bqd
        d = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).cuda()
        self.launches = 1
        if kind in ("nvfp4_encode", "q8_0_encode"):
            M, K = p["M"], p["K"]
            self.w = (d(host["x"]),)  # the bf16 weight being encoded
            self.x_host, self.x = host["x"][:1], self.w[0]
            self.ts = float(self.w[0].view(torch.bfloat16).float().abs().max().item() / (6 * 448))
            if kind == "nvfp4_encode":
                self.out = (torch.empty(M * K // 2, dtype=torch.uint8, device="cuda"),
                            torch.empty(M * K // 16, dtype=torch.uint8, device="cuda"))
            else:
                self.out = (torch.empty(M * K, dtype=torch.int8, device="cuda"),
                            torch.empty(M * K // 32, dtype=torch.int16, device="cuda"))
            self.y = self.out[0]
            self.in_bytes = M * K * 2
        elif kind == "nvfp4_gemm_grouped":
            self.w = (d(host["codes"]), d(host["scales"]))
            self.tse, self.offs = d(host["ts"]), d(host["offsets"])
            self.x_host, self.x = host["x"], d(host["x"])
            self.y = torch.empty(p["N"] * p["M"], dtype=torch.float32, device="cuda")
            self.in_bytes = self.x.numel() * 2
        elif kind in ("nvfp4", "q8_0", "q4_0", "q4_1", "fp8_b128", "nvfp4_tiny", "nvfp4_silu", "nvfp4_add",
                      "nvfp4_gemm"):
            M, K, N = p["M"], p["K"], p["N"]
            if kind == "q8_0":
                self.w = (d(host["q"]), d(host["d"]))
            elif kind == "q4_0":
                self.w = (d(host["codes"]), d(host["d"]))
            elif kind == "q4_1":
                self.w = (d(host["codes"]), d(host["dm"]))
            elif kind == "fp8_b128":
                self.w = (d(host["codes"]), d(host["scales"]))
            else:
                self.w = (d(host["codes"]), d(host["scales"]))
                self.ts = host["ts"]
            self.x_host = host["x"]
            self.x = d(host["x"])
            self.y = torch.empty(N * M, dtype=torch.float32, device="cuda")
            self.in_bytes = self.x.numel() * 2
            if kind == "nvfp4_add":
                self.r = d(host["r"])
                self.in_bytes += self.r.numel() * 4
        else:
            T, E, H, I, k = p["T"], p["E"], p["H"], p["I"], p["topk"]
            self.w = tuple(d(host[n]) for n in ("gu_codes", "gu_scales", "gu_ts", "dn_codes", "dn_scales", "dn_ts"))
            self.x_host, self.logits_host = host["x"], host["logits"]
            self.x, self.logits = d(host["x"]), d(host["logits"])
            if kind == "moe_prefill":
                self.wsb = bqd.moe_prefill_workspace_bytes(T, k, H, I, E)
                self.launches = 6  # route, gather, gate_up GEMM, SiLU * up, down GEMM, combine
            else:
                self.wsb = bqd.moe_layer_workspace_bytes(T, k, H, I, E)
                self.launches = moe_launches(T, E, H, I, k)
            self.ws = torch.empty(self.wsb, dtype=torch.uint8, device="cuda")
            self.y = torch.empty(T * H, dtype=torch.float32, device="cuda")
            self.in_bytes = self.x.numel() * 2 + self.logits.numel() * 4
        self.out_bytes = self.y.numel() * self.y.element_size()
        self.weight_bytes = sum(t.numel() * t.element_size() for t in self.w)
        self.copies = [self.w]

    def make_copies(self, n):
        """n device copies of the weights in all (the original included)."""
        self.copies = [self.w] + [tuple(t.clone() for t in self.w) for _ in range(n - 1)]

    def drop_copies(self):
        self.copies = [self.w]

    def run_path(self, path):
        """The NVFP4 GEMV of this row through an explicit compute path."""
        p = self.p
        self.bqd.nvfp4_gemv_path(self.w[0], self.w[1], self.ts, self.x, self.y, p["M"], p["K"], p["N"], path)

    def run(self, copy=0):
        p, b = self.p, self.bqd
        w = self.copies[copy]
        if self.kind in ("nvfp4", "nvfp4_tiny"):
            b.nvfp4_gemv(w[0], w[1], self.ts, self.x, self.y, p["M"], p["K"], p["N"])
        elif self.kind == "nvfp4_silu":
            b.nvfp4_gemv_silu_mul(w[0], w[1], self.ts, self.x, self.y, p["M"] // 2, p["K"], p["N"])
        elif self.kind == "nvfp4_add":
            b.nvfp4_gemv_add(w[0], w[1], self.ts, self.x, self.r, self.y, p["M"], p["K"], p["N"])
        elif self.kind == "nvfp4_encode":
            b.nvfp4_encode(w[0], self.ts, self.out[0], self.out[1], p["M"], p["K"])
        elif self.kind == "q8_0_encode":
            b.q8_0_encode(w[0], self.out[0], self.out[1], p["M"], p["K"])
        elif self.kind == "q8_0":
            b.q8_0_gemv(w[0], w[1], self.x, self.y, p["M"], p["K"], p["N"])
        elif self.kind == "q4_0":
            b.q4_0_gemv(w[0], w[1], self.x, self.y, p["M"], p["K"], p["N"])
        elif self.kind == "q4_1":
            b.q4_1_gemv(w[0], w[1], self.x, self.y, p["M"], p["K"], p["N"])
        elif self.kind == "fp8_b128":
            b.fp8_b128_gemv(w[0], w[1], self.x, self.y, p["M"], p["K"], p["N"])
        elif self.kind == "nvfp4_gemm":
            b.nvfp4_gemm(w[0], w[1], self.ts, self.x, self.y, p["M"], p["K"], p["N"])
        elif self.kind == "nvfp4_gemm_grouped":
            b.nvfp4_gemm_grouped(w[0], w[1], self.tse, self.x, self.offs, self.y, p["E"], p["M"], p["K"], p["N"])
        elif self.kind == "moe_prefill":
            T, E, H, I, k = p["T"], p["E"], p["H"], p["I"], p["topk"]
            b.moe_prefill_layer(self.logits, *w, self.x, self.y, self.ws, self.wsb, E, H, I, T, k)
        else:
            T, E, H, I, k = p["T"], p["E"], p["H"], p["I"], p["topk"]
            b.moe_layer(self.logits, *w, self.x, self.y, self.ws, self.wsb, E, H, I, T, k)


# ---------------------------------------------------------------- CPU oracle arms
def cpu_units(rows):
    """Per row, a list of (callable, bytes) work units of the fp64 oracle:
    64 weight rows of a GEMV (all N columns), or one routed (token, slot)
    pair of a MoE layer (gate_up, SiLU * up, down for that expert)."""
    import oracle
    out = []
    for name, kind, p, host in rows:
        units = []
        if kind in ("nvfp4", "q8_0"):
            M, K, N = p["M"], p["K"], p["N"]
            for r0 in range(0, M, 64):
                idx = np.arange(r0, min(M, r0 + 64), dtype=np.int64)
                if kind == "nvfp4":
                    f = (lambda idx=idx, h=host, M=M, K=K: oracle.nvfp4_gemv(h["codes"], h["scales"], h["ts"], h["x"],
                                                                           M, K, rows=idx))
                    nb = nvfp4_bytes(len(idx), K, N)
                else:
                    f = lambda idx=idx, h=host, M=M, K=K: oracle.q8_0_gemv(h["q"], h["d"], h["x"], M, K, rows=idx)
                    nb = q8_0_bytes(len(idx), K, N)
                units.append((f, nb))
        else:
            sel, w = oracle.moe_route(host["logits"], p["topk"])
            H, I = p["H"], p["I"]
            for t in range(p["T"]):
                for s in range(p["topk"]):
                    sub = dict(host, T=1, topk=1, x=host["x"][t:t + 1])
                    f = (lambda sub=sub, e=int(sel[t, s]):
                         oracle.moe_layer(sub, sel=np.array([[e]], dtype=np.int32), weights=np.ones((1, 1))))
                    units.append((f, moe_expert_bytes(H, I) + H * 6))
        out.append((name, units))
    return out


def _sample_plan(units, costs, cpu_seconds):
    """The same leading fraction of every row's remaining units, sized so the
    estimated CPU time (per-row unit cost x units) is cpu_seconds."""
    rest = sum(c * (len(u) - 1) for c, (_, u) in zip(costs, units))
    frac = 0.0 if rest <= 0 else max(0.0, min(1.0, cpu_seconds / rest))
    return frac, [1 + int(math.floor((len(u) - 1) * frac)) for _, u in units]


def cpu_baseline_sample(units, budget_s):
    """One host core: the first unit of every row (timed, which gives the
    per-row unit cost) plus the same leading fraction of every row's other
    units, ~budget_s in all. Returns (bytes, seconds, description, costs)."""
    done_b, secs = 0, 0.0
    cost = []
    for _, u in units:
        f, nb = u[0]
        t0 = time.perf_counter()
        f()
        dt = time.perf_counter() - t0
        secs += dt
        done_b += nb
        cost.append(max(dt, 1e-5))
    frac, taken = _sample_plan(units, cost, budget_s - secs)
    for (_, u), take in zip(units, taken):
        for f, nb in u[1:take]:
            t0 = time.perf_counter()
            f()
            secs += time.perf_counter() - t0
            done_b += nb
    desc = (f"fp64 C oracle on 1 host core: the first unit of every row plus the first {frac:.4f} of the "
            f"remaining work units of every row (GEMV unit: 64 weight rows; MoE unit: one routed (token, slot) "
            f"pair); {sum(taken)} of {sum(len(u) for _, u in units)} units")
    return done_b, secs, desc, cost


def cpu_baseline_all_cores(units, costs, budget_s, workers):
    """All host cores: the oracle's work units run by `workers` threads (the
    oracle's C calls release the interpreter lock), the leading fraction of
    every row sized to ~budget_s of wall time. Returns (bytes, wall seconds,
    description)."""
    from concurrent.futures import ThreadPoolExecutor
    frac, taken = _sample_plan(units, costs, budget_s * workers)
    work = [u[i] for (_, u), take in zip(units, taken) for i in range(take)]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda fu: fu[0](), work))
    wall = time.perf_counter() - t0
    desc = (f"fp64 C oracle on {workers} host threads (one per core): the first {frac:.4f} of every row's work "
            f"units (GEMV unit: 64 weight rows; MoE unit: one routed (token, slot) pair); {len(work)} of "
            f"{sum(len(u) for _, u in units)} units")
    return sum(nb for _, nb in work), wall, desc


def host_cpu_info():
    """Core count and CPU model of this host."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
    return {"nproc": os.cpu_count(), "model": model}


def run_reference(args, rank):
    if rank != 0:
        return  # the reference arm runs on rank 0 only
    spec = rows_spec()
    units = cpu_units([(n, k, p, host_inputs(k, p)) for n, k, p in spec])
    per_step = 150.0 / max(1, args.steps + args.warmup)
    cursor = [0] * len(units)

    def step(i):
        r = i % len(units)
        u = units[r][1]
        b, s = 0, 0.0
        while True:
            f, nb = u[cursor[r] % len(u)]
            cursor[r] += 1
            t0 = time.perf_counter()
            f()
            s += time.perf_counter() - t0
            b += nb
            if s >= per_step:
                return b, s

    for i in range(args.warmup):
        step(i)
    tot_b, tot_s = 0, 0.0
    for i in range(args.steps):
        b, s = step(args.warmup + i)
        tot_b += b
        tot_s += s
    value = tot_b / tot_s / 1e9
    desc = (f"fp64 C oracle on 1 host core; each step runs work units (GEMV: 64 weight rows; MoE: one routed "
            f"(token, slot) pair) of one row of the step, rows in turn, for ~{per_step:.3f} s")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; the method's workload shapes)",
            "config": {"workload": WORKLOAD, "sample": desc},
            "cpu_baseline": {"kind": "oracle", "value": value, "unit": "GB/s", "cores": 1, "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist

    import block_quantized_decode_nvfp4_gb300 as bqd
    from block_quantized_decode_nvfp4_gb300 import build as _build

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    bqd.lib()
    bqd.set_launch_flags(bqd.BQD_LAUNCH_PDL if args.launch_pdl == "on" else 0)
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 0) or L2_BYTES_FALLBACK

    spec = rows_spec()
    hosts = {n: host_inputs(k, p, seed=0) for n, k, p in spec}
    rows = [Row(n, k, p, hosts[n], torch, bqd) for n, k, p in spec]
    extra = [Row(n, k, p, host_inputs(k, p, seed=0), torch, bqd) for n, k, p in extra_rows_spec()]
    step_bytes = sum(r.bytes for r in rows)
    launches_per_step = sum(r.launches for r in rows)
    dominant = next(r for r in rows if r.name.startswith("q8_0 151936"))
    stream = torch.cuda.current_stream()

    # warm-up (also performs the library's one-time per-kernel setup)
    for _ in range(max(3, args.warmup)):
        for r in rows + extra:
            r.run()
    torch.cuda.synchronize()

    # ---- per-row isolated timings: L2 emptied by a read-only sweep before each call
    flush = torch.empty(int(2.5 * l2) // 4, dtype=torch.float32, device="cuda").fill_(1.0)

    def isolated_us(fn):
        ts = []
        for i in range(30):
            flush.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if i >= 5:
                ts.append(e0.elapsed_time(e1) * 1e3)  # us
        return statistics.median(ts)

    per_row = [(r, isolated_us(r.run)) for r in rows + extra]

    # ---- per-row back-to-back timings: 200 calls captured in a CUDA graph,
    # cycling through weight copies whose calls' working set exceeds 3x L2
    def back_to_back_us(r, n_calls=200, reps=10):
        R = rotating_copies(r.bytes, r.weight_bytes, l2, args.copy_budget_gb * 1e9)
        r.make_copies(R)
        for i in range(R):
            r.run(i)
        torch.cuda.synchronize()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            for i in range(n_calls):
                r.run(i % R)
        ts = []
        with torch.cuda.stream(cs):
            for rep in range(reps + 2):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(cs)
                g.replay()
                e1.record(cs)
                e1.synchronize()
                if rep >= 2:
                    ts.append(e0.elapsed_time(e1) * 1e3 / n_calls)
        del g
        r.drop_copies()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        return statistics.median(ts), R

    b2b = {r.name: back_to_back_us(r) for r in rows + extra}
    # the multi-token (verify) rows through the CUDA-core, tcgen05 and warp-tile paths
    verify_paths = {}
    for r in rows:
        if r.kind == "nvfp4" and r.p["N"] > 1:
            cc = isolated_us(lambda r=r: r.run_path(bqd.BQD_PATH_CUDA_CORE))
            mma = isolated_us(lambda r=r: r.run_path(bqd.BQD_PATH_MMA))
            tiles = isolated_us(lambda r=r: r.run_path(bqd.BQD_PATH_TILES))
            verify_paths[r.name] = {"cuda_core_us": round(cc, 3), "mma_us": round(mma, 3),
                                    "tiles_us": round(tiles, 3), "mma_GB_s": round(r.bytes / mma / 1e3, 1),
                                    "speedup": round(cc / mma, 3)}

    # ---- headline: K full steps, inputs resident in HBM
    peak, peak_kind = measured_peaks()
    tensor_peak = measured_tensor_peak()
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    dom_events = []
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        for r in rows:
            if r is dominant:
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                r.run()
                b_.record(stream)
                dom_events.append((a, b_))
            else:
                r.run()
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    elapsed_s = max_over_ranks(t_start.elapsed_time(t_end) / 1e3, world, "cuda")
    dom_us = statistics.mean(a.elapsed_time(b_) * 1e3 for a, b_ in dom_events)

    # ---- e2e: host buffers through the public API, copies inside the timed region
    pinned_in, pinned_out = [], []
    for r in rows:
        xs = [torch.from_numpy(r.x_host.view(np.int16)).pin_memory()]
        if r.kind == "moe":
            xs.append(torch.from_numpy(r.logits_host).pin_memory())
        pinned_in.append(xs)
        pinned_out.append(torch.empty(r.y.numel(), dtype=torch.float32).pin_memory())
    h2d = sum(r.in_bytes for r in rows)
    d2h = sum(r.out_bytes for r in rows)
    e2e_steps = max(3, min(args.steps, 200))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for r, xs, yo in zip(rows, pinned_in, pinned_out):
            r.x.copy_(xs[0], non_blocking=True)
            if r.kind == "moe":
                r.logits.copy_(xs[1], non_blocking=True)
            r.run()
            yo.copy_(r.y, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world, "cuda")

    # ---- CPU baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        units = cpu_units([(r.name, r.kind, r.p, hosts[r.name]) for r in rows])
        b1, s1, desc1, costs = cpu_baseline_sample(units, args.cpu_budget)
        info = host_cpu_info()
        workers = info["nproc"] or 1
        bn, sn, descn = cpu_baseline_all_cores(units, costs, args.cpu_budget, workers)
        cpu = {"value": bn / sn / 1e9, "unit": "GB/s", "cores": workers, "kind": "oracle", "sample": descn,
               "single_core": {"value": b1 / s1 / 1e9, "unit": "GB/s", "cores": 1, "sample": desc1},
               "host": info}

    if rank != 0:
        return
    ms = elapsed_s / args.steps * 1e3
    value = whole_job_gbs(step_bytes, world, args.steps, elapsed_s)
    traffic = profiled_traffic(dominant.name)
    breakdown = {}
    for r, us in per_row:
        gbs = r.bytes / us / 1e3
        bus, copies = b2b[r.name]
        bgbs = r.bytes / bus / 1e3
        ent = {"us_per_call": round(us, 3), "GB_s": round(gbs, 1), "frac_hbm": round(gbs / peak, 4),
               "b2b_us_per_call": round(bus, 3), "b2b_GB_s": round(bgbs, 1), "b2b_frac_hbm": round(bgbs / peak, 4),
               "b2b_weight_copies": copies, "bytes": r.bytes, "in_step": r in rows}
        tr = profiled_traffic(r.name)
        ent["traffic"] = tr
        ent["traffic_ratio"] = None if tr is None else round(tr / r.bytes, 4)
        if r.kind in ("nvfp4_gemm", "nvfp4_gemm_grouped", "moe_prefill"):  # flops against the bf16 tensor peak
            fl = (2.0 * r.p["M"] * r.p["K"] * r.p["N"] if r.kind != "moe_prefill"
                  else 2.0 * r.p["T"] * r.p["topk"] * 3 * r.p["H"] * r.p["I"])
            ent["TFLOP_s"] = round(fl / us / 1e6, 1)
            ent["b2b_TFLOP_s"] = round(fl / bus / 1e6, 1)
            ent["frac_tensor"] = round(fl / bus / 1e6 / tensor_peak, 4)
            ent["tensor_peak_TFLOP_s"] = tensor_peak
        if r.kind in ("moe", "moe_prefill"):
            ent["us_per_token"] = round(us / r.p["T"], 3)
            ent["b2b_us_per_token"] = round(bus / r.p["T"], 3)
            ent["tokens_per_s"] = round(r.p["T"] * 1e6 / us, 1)
            ent["b2b_tokens_per_s"] = round(r.p["T"] * 1e6 / bus, 1)
        else:
            ent["tokens_per_s_equiv"] = round(r.p["N"] * 1e6 / us, 1)
            ent["b2b_tokens_per_s_equiv"] = round(r.p["N"] * 1e6 / bus, 1)
        breakdown[r.name] = ent
    dom_gbs = dominant.bytes / dom_us / 1e3
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; the method's workload shapes)",
        "config": {"workload": WORKLOAD, "step_bytes": step_bytes, "launch_pdl": args.launch_pdl,
                   "l2": f"inputs larger than L2: one step streams {step_bytes / 1e9:.2f} GB vs L2 "
                         f"{l2 / 2**20:.0f} MiB; per-row isolated figures flush L2 with a read sweep before "
                         f"each call; per-row back-to-back figures replay 200 graph-captured calls cycling "
                         f"through weight copies whose calls stream more than 3x L2",
                   "formats": "NVFP4 (E2M1 + E4M3/16 + fp32 ts), Q8_0 (int8 + fp16/32); bf16 x; fp32 accumulate"},
        "roofline": {"bound": "hbm", "kernel": dominant.name, "achieved": round(dom_gbs, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(dom_gbs / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": dominant.bytes},
        "rows": breakdown,
        "verify_paths": verify_paths,
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "e2e": {"value": round(whole_job_gbs(step_bytes, world, 1, e2e_s), 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 4),
                "note": "weights resident (model parameters); per step: pinned H2D of every row's "
                        "activations and router logits, all calls, D2H of every output, stream sync"},
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_profile_row(args):
    """Call one row of the step a few times and nothing else (for ncu)."""
    import torch

    import block_quantized_decode_nvfp4_gb300 as bqd
    from block_quantized_decode_nvfp4_gb300 import build as _build

    _build.build()
    spec = {n: (k, p) for n, k, p in rows_spec() + extra_rows_spec()}
    if args.profile_row not in spec:
        raise SystemExit(f"unknown row {args.profile_row!r}; rows: {sorted(spec)}")
    kind, p = spec[args.profile_row]
    row = Row(args.profile_row, kind, p, host_inputs(kind, p), torch, bqd)
    for _ in range(args.profile_calls):
        row.run()
    torch.cuda.synchronize()


# Kernel sources each row's DRAM record depends on (a record is used only
# while these files are unchanged).
TRAFFIC_SOURCES = {
    "direct": ["gemv_direct.cu", "common.cuh", "gemv.h", "host_util.h"],
    "mma": ["gemv_mma.cu", "common.cuh", "stream.cuh", "gemv.h", "host_util.h"],
    "stream": ["gemv_stream.cu", "common.cuh", "stream.cuh", "gemv.h", "host_util.h"],
    "moe": ["moe_small.cu", "moe_route.cuh", "common.cuh", "stream.cuh", "gemv.h", "host_util.h"],
    "encode": ["encode.cu", "common.cuh", "gemv.h", "host_util.h"],
    "gemm": ["gemm_prefill.cu", "gemm.h", "common.cuh", "stream.cuh", "host_util.h"],
    "moe_prefill": ["moe_prefill.cu", "moe_route.cuh", "gemm_prefill.cu", "gemm.h", "common.cuh", "stream.cuh",
                    "gemv.h", "host_util.h"],
}


def traffic_sources(kind, p):
    if kind == "moe":
        return TRAFFIC_SOURCES["moe"]
    if kind.endswith("encode"):
        return TRAFFIC_SOURCES["encode"]
    if kind in ("nvfp4_gemm", "nvfp4_gemm_grouped"):
        return TRAFFIC_SOURCES["gemm"]
    if kind == "moe_prefill":
        return TRAFFIC_SOURCES["moe_prefill"]
    if p.get("N", 1) > 1:
        return TRAFFIC_SOURCES["mma"]
    return TRAFFIC_SOURCES["stream" if p["K"] % 1024 else "direct"]


SEPARATOR_KERNEL = "nvfp4_dequant_kernel"  # launched between rows by --profile-all; no row uses it


def write_traffic(csv_path, calls, out_path=None):
    """profiles/traffic.json from the ncu CSV (dram__bytes_read.sum,
    dram__bytes_write.sum) of `bench.py --profile-all --profile-calls
    <calls>`: the launches are split into rows at the separator kernel,
    torch's own kernels (the rows' setup) are left out, and each row's bytes
    are divided by the number of calls."""
    import csv
    spec = rows_spec() + extra_rows_spec()
    with open(csv_path) as f:
        recs = [r for r in csv.reader(f) if len(r) > 10]
    h = recs[0]
    ki, mi, vi, ii = (h.index(c) for c in ("Kernel Name", "Metric Name", "Metric Value", "ID"))
    launches = {}
    for r in recs[1:]:
        launches.setdefault(int(r[ii]), {"k": r[ki]})[r[mi]] = float(r[vi].replace(",", ""))
    segs = None
    for _, v in sorted(launches.items()):
        name = v["k"]
        if SEPARATOR_KERNEL in name:
            segs = [] if segs is None else segs
            segs.append([])
        elif segs is not None and not (name.startswith("void at::") or name.startswith("at::")):
            segs[-1].append(v)
    if segs is None or len(segs) != len(spec):
        raise SystemExit(f"{0 if segs is None else len(segs)} row segments in {csv_path}, {len(spec)} rows expected")
    out = {}
    for (row, kind, p), seg in zip(spec, segs):
        rd = sum(v["dram__bytes_read.sum"] for v in seg) / calls
        wr = sum(v["dram__bytes_write.sum"] for v in seg) / calls
        kern = sorted({v["k"].split("(")[0].replace("void ", "").replace("bqd::", "").replace("<unnamed>::", "")
                       .replace("(anonymous namespace)::", "") for v in seg})
        alg = row_bytes(kind, p, host_inputs(kind, p) if kind in ("moe", "moe_prefill") else None)
        src = traffic_sources(kind, p)
        out[row] = {"source_sha": source_sha(src), "sources": src, "kernels": kern,
                    "launches_per_call": len(seg) // calls, "dram_bytes_per_launch": int(round(rd + wr)),
                    "dram_read": int(round(rd)), "dram_write": int(round(wr)), "algorithmic_bytes": int(alg),
                    "ratio": round((rd + wr) / alg, 4)}
        print(f"{row:52s} {out[row]['dram_bytes_per_launch']:>12d} alg {alg:>12d} ratio {out[row]['ratio']}")
    with open(out_path or os.path.join(ROOT, "profiles", "traffic.json"), "w") as f:
        json.dump(out, f, indent=1)


def run_profile_all(args):
    """Every row (step rows, then extra rows) called --profile-calls times
    and nothing else, a separator launch before each row; for a per-row ncu
    capture in one process (see write_traffic)."""
    import torch

    import block_quantized_decode_nvfp4_gb300 as bqd
    from block_quantized_decode_nvfp4_gb300 import build as _build

    _build.build()
    rows = [Row(n, k, p, host_inputs(k, p), torch, bqd) for n, k, p in rows_spec() + extra_rows_spec()]
    sc = torch.zeros(16 * 8, dtype=torch.uint8, device="cuda")
    ss = torch.zeros(16, dtype=torch.uint8, device="cuda")
    sw = torch.empty(16 * 16, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for r in rows:
        bqd.nvfp4_dequant(sc, ss, 1.0, sw, 16, 16)
        for _ in range(args.profile_calls):
            r.run()
    torch.cuda.synchronize()


def run_profile_step(args):
    """Run --steps decode steps (every row once per step, in step order) and
    nothing else: the launch list of the timed region, for profilers."""
    import torch

    import block_quantized_decode_nvfp4_gb300 as bqd
    from block_quantized_decode_nvfp4_gb300 import build as _build

    _build.build()
    bqd.set_launch_flags(bqd.BQD_LAUNCH_PDL if args.launch_pdl == "on" else 0)
    rows = [Row(n, k, p, host_inputs(k, p, seed=0), torch, bqd) for n, k, p in rows_spec()]
    for _ in range(args.steps):
        for r in rows:
            r.run()
    torch.cuda.synchronize()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--copy-budget-gb", type=float, default=40.0,
                    help="device memory for the weight copies of one row's back-to-back timing")
    ap.add_argument("--launch-pdl", choices=["on", "off"], default="on",
                    help="programmatic dependent launch between the step's kernels (BQD_LAUNCH_PDL)")
    ap.add_argument("--profile-row", default=None,
                    help="only call this row of the step (e.g. 'q8_0 151936x4096 N=1') --profile-calls times, "
                         "for profilers; prints no JSON line")
    ap.add_argument("--profile-calls", type=int, default=3)
    ap.add_argument("--profile-step", action="store_true",
                    help="only run --steps decode steps (no per-row timings, no JSON line), for profilers")
    ap.add_argument("--profile-all", action="store_true",
                    help="call every row --profile-calls times, a separator launch before each (for ncu)")
    ap.add_argument("--write-traffic", default=None, metavar="CSV",
                    help="write profiles/traffic.json from the ncu CSV of --profile-all (no GPU needed)")
    ap.add_argument("--list-rows", action="store_true", help="print the names of every row, one per line")
    args = ap.parse_args()
    if args.list_rows:
        for n, _, _ in rows_spec() + extra_rows_spec():
            print(n)
        return
    if args.write_traffic is not None:
        write_traffic(args.write_traffic, args.profile_calls)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.profile_row is not None:
        run_profile_row(args)
        return
    if args.profile_all:
        run_profile_all(args)
        return
    if args.profile_step:
        run_profile_step(args)
        return
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
