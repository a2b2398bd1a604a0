#!/usr/bin/env python3
"""Benchmark of the k-quant x q8_1 contraction on GB300.

One "step" is one pass of the whole hot path over one batch of synthetic
input: q8_1 quantization of every distinct activation, then the GEMV (decode)
or MMQ (prefill) of every weight that reads it, residual adds fused.

Workloads (benchmark configurations; shapes of the named models, synthetic
data of the stated distributions):
  0  single Q4_K GEMV 4096 x 4096, M = 1
  1  Llama-3-8B decode layer, M = 1: QKV 6144x4096, attn-out 4096x4096 (+res),
     gate||up 28672x4096 (one q8_1 activation), down 4096x14336 (+res)   [default]
  2  Q6_K output head 128256 x 4096, M = 1
  3  config 1 + config 2 at M = 4
  4  Qwen2-7B prefill MMQ at M = 2048: QKV 4608x3584, attn-out 3584x3584 (+res),
     gate||up 37888x3584, down 3584x18944 (+res)
  5  config 4 as a Q4_K_M layer that keeps its down projection in Q6_K (the
     Q4_K_M recipe routes some down and value projections to Q6_K)
  6  config 1 as a chain with the fused producers: RMSNorm -> q8_1 feeds QKV,
     attn-out adds the residual stream h, RMSNorm(h) -> q8_1 feeds gate||up,
     SwiGLU -> q8_1 of its output feeds down, which adds h (attention itself is
     not part of the path: its output is a synthetic input)
  7  config 1 with every weight in Q5_K (a Q5_K_M-style layer)
  8  config 1 with every weight in Q8_0
  9  config 1 with every weight in Q3_K
 10  config 1 with every weight in Q2_K

Timing: W untimed warm-up steps, then exactly K steps replayed from CUDA
graphs (programmatic dependent launch between the kernels), bracketed by a
barrier and torch.cuda.synchronize(), timed with CUDA events on the launching
stream.  Weight copies rotate between steps so the working set exceeds L2.
`--impl reference` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Q4_K/Q6_K GEMV weight GB/s (% of HBM peak); prefill MMQ int8 TOPS"
L2_BYTES = 129 * 2 ** 20
# device bytes per 256 weights (GGUF bytes, except Q3_K whose scales the repack unpacks: 114 for 110)
BYTES_PER_SB = {"q4k": 144, "q6k": 210, "q5k": 176, "q80": 272, "q2k": 84, "q3k": 114}
OTYPE = {"q4k": 1, "q6k": 2, "q5k": 3, "q80": 4, "q2k": 5, "q3k": 6}   # type ids (library and oracle)

CONFIGS = {
    0: dict(name="single Q4_K GEMV 4096x4096, batch 1", M=1, kind="gemv",
            gemms=[("w", "q4k", 4096, 4096, False, "x")]),
    1: dict(name="Llama-3-8B decode layer, batch 1 (Q4_K)", M=1, kind="gemv",
            gemms=[(n, "q4k", N, K, r, s) for (n, N, K, r, s) in synth.LLAMA3_8B_LAYER]),
    2: dict(name="Q6_K output head 128256x4096, batch 1", M=1, kind="gemv",
            gemms=[("head", "q6k", 128256, 4096, False, "x_head")]),
    3: dict(name="Llama-3-8B decode layer + Q6_K head, 4 sequences", M=4, kind="gemv",
            gemms=[(n, "q4k", N, K, r, s) for (n, N, K, r, s) in synth.LLAMA3_8B_LAYER]
            + [("head", "q6k", 128256, 4096, False, "x_head")]),
    4: dict(name="Qwen2-7B prefill MMQ, 2048 tokens (Q4_K)", M=2048, kind="mmq",
            gemms=[(n, "q4k", N, K, r, s) for (n, N, K, r, s) in synth.QWEN2_7B_PREFILL]),
    5: dict(name="Qwen2-7B prefill MMQ, 2048 tokens (Q4_K, down projection in Q6_K)", M=2048, kind="mmq",
            gemms=[(n, "q6k" if n == "down" else "q4k", N, K, r, s) for (n, N, K, r, s) in synth.QWEN2_7B_PREFILL]),
    6: dict(name="Llama-3-8B decode layer with fused RMSNorm/SwiGLU -> q8_1 producers, batch 1 (Q4_K)", M=1,
            kind="chain", gemms=[(n, "q4k", N, K, r, s) for (n, N, K, r, s) in synth.LLAMA3_8B_LAYER],
            inputs=["x_attn_in", "x_attn_out"]),
    7: dict(name="Llama-3-8B decode layer, batch 1 (Q5_K)", M=1, kind="gemv",
            gemms=[(n, "q5k", N, K, r, s) for (n, N, K, r, s) in synth.LLAMA3_8B_LAYER]),
    8: dict(name="Llama-3-8B decode layer, batch 1 (Q8_0)", M=1, kind="gemv",
            gemms=[(n, "q80", N, K, r, s) for (n, N, K, r, s) in synth.LLAMA3_8B_LAYER]),
    9: dict(name="Llama-3-8B decode layer, batch 1 (Q3_K)", M=1, kind="gemv",
            gemms=[(n, "q3k", N, K, r, s) for (n, N, K, r, s) in synth.LLAMA3_8B_LAYER]),
    10: dict(name="Llama-3-8B decode layer, batch 1 (Q2_K)", M=1, kind="gemv",
             gemms=[(n, "q2k", N, K, r, s) for (n, N, K, r, s) in synth.LLAMA3_8B_LAYER]),
}
NORM_EPS = 1e-5                                       # Llama-3 RMSNorm epsilon


def weight_bytes(cfg) -> int:
    return sum(N * (K // 256) * BYTES_PER_SB[q] for (_, q, N, K, _, _) in cfg["gemms"])


def int_ops(cfg) -> int:
    return sum(2 * cfg["M"] * N * K for (_, _, N, K, _, _) in cfg["gemms"])


def gemm_fused(policy: str, cfg, gemm) -> bool:
    if cfg["kind"] == "chain":                      # only attn-out reads an f32 activation the chain does not make
        return gemm[0] == "attn_out"
    """Decode activation path of one GEMM: q8_1 quantization inside the GEMV ("fused")
    or a quantize kernel before its consumers.  "auto" quantizes inside the GEMV when the
    activation is small (M*K <= 4096: one float4 or two per thread), where saving the
    extra kernel and dependency wins; larger activations use the quantize kernel, since
    the in-GEMV front end repeats the quantization in every CTA."""
    if cfg["kind"] != "gemv":
        return False
    if policy == "auto":
        return cfg["M"] * gemm[3] <= 4096
    return policy == "fused"


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, averaged over the
# kernel's launches in one step) from one ncu capture of the command in the named profile.
# Valid only while the kernel sources are the ones the counters were taken on.
TRAFFIC: dict = {
    (1, "gemv_q4k_f32"): {"bytes_per_launch": 29981181, "digest": "bc3a9e2fedd8c4ef",
                          "profile": "profiles/dram_traffic_per_launch.md"},
    (2, "gemv_q6k_f32"): {"bytes_per_launch": 437107968, "digest": "bc3a9e2fedd8c4ef",
                          "profile": "profiles/gemv_q6k_f32_head_128256x4096.md"},
    (3, "gemv_q6k"): {"bytes_per_launch": 435261696, "digest": "bc3a9e2fedd8c4ef",
                      "profile": "profiles/dram_traffic_per_launch.md"},
    (4, "mmq_q4k"): {"bytes_per_launch": 233749376, "digest": "b1c1938ee3b443a4",
                     "profile": "profiles/dram_traffic_per_launch.md"},
}


def front_end_desc(front_end: str, cfg) -> str:
    if cfg["kind"] == "chain":
        return ("producers: qk_rmsnorm_q8_1 -> qkv; attn_out quantizes its f32 input inside the GEMV; "
                "qk_rmsnorm_q8_1 -> gate_up; qk_swiglu_q8_1 -> down")
    if cfg["kind"] != "gemv":
        return "qk_quantize_q8_1 kernel per activation"
    parts = []
    for g in cfg["gemms"]:
        parts.append(f"{g[0]}: " + ("q8_1 quantization inside the GEMV" if gemm_fused(front_end, cfg, g)
                                     else "qk_quantize_q8_1 kernel"))
    return f"{front_end}: " + "; ".join(parts)


# the sources a kernel family is compiled from; a recorded traffic figure holds while they are unchanged
KERNEL_SOURCES = {"gemv": ("qk_common.cuh", "qk_gemv.cu"), "mmq": ("qk_common.cuh", "qk_tc.cuh", "qk_mmq.cu")}


def kernel_sources_digest(kernel: str) -> str:
    import hashlib
    d = hashlib.sha1()
    src = os.path.join(ROOT, "quantized_q8_activation_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel.split("_")[0]]:
        d.update(f.encode())
        with open(os.path.join(src, f), "rb") as fh:
            d.update(fh.read())
    return d.hexdigest()[:16]


def recorded_traffic(cfg_id: int, kernel: str):
    t = TRAFFIC.get((cfg_id, kernel))
    if t is None or t["digest"] != kernel_sources_digest(kernel):
        return None
    return t["bytes_per_launch"]


def launches_per_step(cfg, front_end: str = "auto") -> int:
    """kernels of this library one step launches: the quantize kernels of unfused activations,
    one GEMV per decode GEMM, two kernels (prep and main) per MMQ call, and the chain's
    two RMSNorm and one SwiGLU producers"""
    if cfg["kind"] == "chain":
        return 3 + len(cfg["gemms"])
    slots_q = {g[5] for g in cfg["gemms"] if not gemm_fused(front_end, cfg, g)}
    per_gemm = 2 if cfg["kind"] == "mmq" else 1
    return len(slots_q) + per_gemm * len(cfg["gemms"])


def slots(cfg):
    """activation slots in step order with their K"""
    out = []
    for (_, _, _, K, _, s) in cfg["gemms"]:
        if s not in [a for a, _ in out]:
            out.append((s, K))
    return out


# ------------------------------------------------------------------ workload

class Workload:
    """Device buffers for one configuration: repacked weights (several copies),
    f32 activations and residuals, q8_1 buffers and outputs."""

    def __init__(self, cfg_id: int, seed: int = 0, copies: int | None = None, device="cuda"):
        import quantized_q8_activation_gb300 as qk
        self.qk = qk
        self.cfg_id = cfg_id
        self.cfg = cfg = CONFIGS[cfg_id]
        self.M = M = cfg["M"]
        wb = weight_bytes(cfg)
        if copies is None:
            copies = max(1, -(-3 * L2_BYTES // wb))         # working set >= 3 x L2
        self.copies = copies
        self.host_w, self.w = {}, [dict() for _ in range(copies)]
        for (name, q, N, K, _, _) in cfg["gemms"]:
            hw = synth.weights(q, N, K, seed=seed, tag=name)
            self.host_w[name] = hw
            g = torch.from_numpy(hw).to(device)
            for c in range(copies):
                self.w[c][name] = qk.repack(OTYPE[q], g, N, K)
            del g
        self.host_x = {s: synth.activations(M, K, seed=seed, tag=s) for s, K in slots(cfg)
                       if s in cfg.get("inputs", [s])}
        self.x = {s: torch.from_numpy(v).to(device) for s, v in self.host_x.items()}
        self.q8 = {s: qk.empty_q8_1(M, K, device) for s, K in slots(cfg)}
        self.host_r, self.r, self.y = {}, {}, {}
        for (name, _, N, _, res, _) in cfg["gemms"]:
            if res:
                self.host_r[name] = synth.residual(M, N, seed=seed, tag=name)
                self.r[name] = torch.from_numpy(self.host_r[name]).to(device)
            self.y[name] = torch.empty((M, N), dtype=torch.float32, device=device)
        self.host_g = {}
        if cfg["kind"] == "chain":
            self.host_g = chain_norm_weights(cfg, seed)
            self.g = {t: torch.from_numpy(v).to(device) for t, v in self.host_g.items()}
            self.r["down"] = self.y["attn_out"]       # down adds the residual stream h = attn-out's output
            del self.host_r["down"]
        self.ws = None
        if cfg["kind"] == "mmq":
            need = max(qk.mmq_workspace_bytes(M, N, K) for (_, _, N, K, _, _) in cfg["gemms"])
            self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device) if need else None
        torch.cuda.synchronize()

    def launch(self, gemm, copy: int, pdl: bool = True, stream=None, fused: bool = True):
        """Enqueue the contraction kernel of one GEMM of the step (its q8_1 input, if it
        has one, must already be in self.q8)."""
        qk, cfg = self.qk, self.cfg
        name, q, N, K, res, s = gemm
        if fused and cfg["kind"] in ("gemv", "chain"):
            fn = {"q4k": qk.gemv_q4k_f32, "q5k": qk.gemv_q5k_f32, "q6k": qk.gemv_q6k_f32, "q80": qk.gemv_q8_0_f32,
                  "q2k": qk.gemv_q2k_f32, "q3k": qk.gemv_q3k_f32}[q]
            fn(self.w[copy][name], self.x[s], N, K, residual=self.r.get(name), y=self.y[name],
               pdl=pdl, stream=stream)
        else:
            codes, scales = self.q8[s]
            kw = dict(residual=self.r.get(name), y=self.y[name], pdl=pdl, stream=stream)
            if cfg["kind"] == "mmq":
                fn = qk.mmq_q4k if q == "q4k" else qk.mmq_q6k
                fn(self.w[copy][name], codes, scales, N, K, workspace=self.ws, **kw)
            else:
                fn = {"q4k": qk.gemv_q4k, "q5k": qk.gemv_q5k, "q6k": qk.gemv_q6k, "q80": qk.gemv_q8_0,
                      "q2k": qk.gemv_q2k, "q3k": qk.gemv_q3k}[q]
                fn(self.w[copy][name], codes, scales, N, K, **kw)

    def step(self, copy: int, pdl: bool = True, stream=None, front_end: str = "auto"):
        """Enqueue one step on `stream`.  Each decode GEMM either quantizes its activation
        inside the GEMV (qk_gemv_*_f32) or reads the q8_1 codes of a quantize kernel that
        runs once per activation before its first consumer (see gemm_fused)."""
        qk, cfg = self.qk, self.cfg
        if cfg["kind"] == "chain":
            return self.chain_step(copy, pdl, stream)
        done = set()
        for gemm in cfg["gemms"]:
            s = gemm[5]
            fused = gemm_fused(front_end, cfg, gemm)
            if not fused and s not in done:
                codes, scales = self.q8[s]
                qk.quantize_q8_1(self.x[s], codes, scales, pdl=pdl, stream=stream)
                done.add(s)
            self.launch(gemm, copy, pdl=pdl, stream=stream, fused=fused)

    def chain_step(self, copy: int, pdl: bool, stream):
        """The decode layer with its producers: RMSNorm -> q8_1 -> QKV; attn-out (+ residual
        stream) -> h; RMSNorm(h) -> q8_1 -> gate||up; SwiGLU -> q8_1 -> down (+ h)."""
        qk, g = self.qk, {gm[0]: gm for gm in self.cfg["gemms"]}
        kw = dict(pdl=pdl, stream=stream)
        c, s = self.q8["x_attn_in"]
        qk.rmsnorm_q8_1(self.x["x_attn_in"], self.g["attn"], NORM_EPS, codes=c, scales=s, **kw)
        self.launch(g["qkv"], copy, fused=False, **kw)
        self.launch(g["attn_out"], copy, fused=True, **kw)
        c, s = self.q8["x_ffn_in"]
        qk.rmsnorm_q8_1(self.y["attn_out"], self.g["ffn"], NORM_EPS, codes=c, scales=s, **kw)
        self.launch(g["gate_up"], copy, fused=False, **kw)
        c, s = self.q8["x_ffn_mid"]
        qk.swiglu_q8_1(self.y["gate_up"], g["gate_up"][2] // 2, codes=c, scales=s, **kw)
        self.launch(g["down"], copy, fused=False, **kw)

    def kernel_key(self, gemm, fused: bool) -> str:
        q = gemm[1]
        if self.cfg["kind"] == "mmq":
            return "mmq_q4k" if q == "q4k" else "mmq_q6k"
        return "gemv_" + q + ("_f32" if fused else "")

    def launches_per_step(self, front_end: str = "auto") -> int:
        return launches_per_step(self.cfg, front_end)


# -------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.dev)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        else:
            self.lines = []

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# -------------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier_max(value: float, ws: int, device):
    if ws == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle

def sample_rows(N: int, n_frac: float) -> int:
    return max(1, min(N, int(round(N * n_frac))))


def chain_norm_weights(cfg, seed: int = 0):
    K = cfg["gemms"][0][3]
    return {t: synth.norm_weight(K, seed=seed, tag=t) for t in ("attn", "ffn")}


def oracle_chain_step(cfg, host_w, host_x, host_r, host_g, threads: int, n_frac: float = 1.0):
    """The decode chain with its producers on the CPU oracle (RMSNorm, q8_1, contraction, SwiGLU),
    each contraction on its first n_frac of output rows (the rest of its output left zero)."""
    import oracle
    gm = {g[0]: g for g in cfg["gemms"]}
    M = cfg["M"]
    units = 0

    def gemm(name, x32, residual):
        nonlocal units
        _, q, N, K, _, _ = gm[name]
        c, d, _ = oracle.quantize_q8_1(x32)
        n1 = sample_rows(N, n_frac)
        y, _ = oracle.gemm(OTYPE[q], host_w[name], N, K, c, d,
                           residual=residual, rows=(0, n1), threads=threads)
        out = np.zeros((M, N), np.float32)
        out[:, :n1] = y
        units += n1 * (K // 256) * BYTES_PER_SB[q]
        return out

    y1, _ = oracle.rmsnorm(host_x["x_attn_in"], host_g["attn"], NORM_EPS)
    gemm("qkv", y1.astype(np.float32), None)
    h = gemm("attn_out", host_x["x_attn_out"], host_r["attn_out"])
    y2, _ = oracle.rmsnorm(h, host_g["ffn"], NORM_EPS)
    gu = gemm("gate_up", y2.astype(np.float32), None)
    mid = oracle.swiglu(gu, gm["gate_up"][2] // 2).astype(np.float32)
    gemm("down", mid, h)
    return units


def oracle_step(cfg, host_w, host_x, host_r, threads: int, m_rows=None, n_frac: float = 1.0, host_g=None):
    """One step of the workload on the CPU oracle (quantize + every contraction).
    m_rows limits the activation rows and n_frac the output rows of every contraction
    (bounded samples); returns the units (weight bytes or int ops) the sample covers."""
    if cfg["kind"] == "chain":
        return oracle_chain_step(cfg, host_w, host_x, host_r, host_g, threads, n_frac)
    import oracle
    q8 = {}
    for s, x in host_x.items():
        xx = x if m_rows is None else x[:m_rows]
        c, d, _ = oracle.quantize_q8_1(xx)
        q8[s] = (c, d)
    wbytes = ops = 0
    for (name, q, N, K, res, s) in cfg["gemms"]:
        c, d = q8[s]
        r = host_r.get(name)
        if r is not None and m_rows is not None:
            r = r[:m_rows]
        n1 = sample_rows(N, n_frac)
        oracle.gemm(OTYPE[q], host_w[name], N, K, c, d, residual=r,
                    rows=(0, n1), threads=threads)
        wbytes += n1 * (K // 256) * BYTES_PER_SB[q]
        ops += 2 * c.shape[0] * n1 * K
    return ops if cfg["kind"] == "mmq" else wbytes


def cpu_baseline(wl_host, cfg, budget_s: float = 12.0, host_g=None):
    """Time the oracle as it stands on the host cores; bounded sample."""
    threads = os.cpu_count() or 1
    host_w, host_x, host_r = wl_host
    if cfg["kind"] == "mmq":
        m_rows = 8                                      # 8 of the 2048 tokens per sample step
        unit, scale = "TOPS", 1e12
        sample = f"{m_rows} of {cfg['M']} activation rows of every GEMM per step (quantize + contraction)"
    else:
        m_rows = None
        unit, scale = "GB/s", 1e9
        sample = ("the full step (quantize + every contraction" +
                  (", RMSNorm and SwiGLU" if cfg["kind"] == "chain" else "") + ") per sample")
    t0 = time.perf_counter()
    n = 0
    done = 0
    while True:
        done += oracle_step(cfg, host_w, host_x, host_r, threads, m_rows, host_g=host_g)
        n += 1
        if time.perf_counter() - t0 >= budget_s or n >= 100000:
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt / scale, "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"{n} x {sample}; {dt:.1f} s"}


# ----------------------------------------------------------------- main arms

def run_reference(args, ws, rank):
    """The oracle on the host cores, on our arm's config/metric/unit.  Each step is a
    bounded sample of the workload (every contraction on a slice of its output rows, and
    for the prefill config on 8 activation rows), sized so the whole run takes about
    --ref-seconds (two minutes by default) whatever --steps is."""
    if rank != 0:
        return
    cfg = CONFIGS[args.config]
    host_w = {name: synth.weights(q, N, K, seed=0, tag=name) for (name, q, N, K, _, _) in cfg["gemms"]}
    host_x = {s: synth.activations(cfg["M"], K, seed=0, tag=s) for s, K in slots(cfg) if s in cfg.get("inputs", [s])}
    host_r = {name: synth.residual(cfg["M"], N, seed=0, tag=name) for (name, _, N, _, res, _) in cfg["gemms"] if res}
    host_g = chain_norm_weights(cfg) if cfg["kind"] == "chain" else None
    threads = os.cpu_count() or 1
    m_rows = 8 if cfg["kind"] == "mmq" else None
    # calibrate on a 1/64 slice, then size the per-step slice to the time budget
    t0 = time.perf_counter()
    oracle_step(cfg, host_w, host_x, host_r, threads, m_rows, n_frac=1 / 64, host_g=host_g)
    t_slice = max(time.perf_counter() - t0, 1e-4)
    per_step = args.ref_seconds / (args.steps + args.warmup)
    n_frac = min(1.0, max(1e-6, per_step / (t_slice * 64)))
    for _ in range(args.warmup):
        oracle_step(cfg, host_w, host_x, host_r, threads, m_rows, n_frac, host_g=host_g)
    t0 = time.perf_counter()
    units = 0
    for _ in range(args.steps):
        units += oracle_step(cfg, host_w, host_x, host_r, threads, m_rows, n_frac, host_g=host_g)
    dt = time.perf_counter() - t0
    if cfg["kind"] == "mmq":
        value, unit = units / dt / 1e12, "TOPS"
        sample = f"{m_rows} of {cfg['M']} activation rows"
    else:
        value, unit = units / dt / 1e9, "GB/s"
        sample = "all activation rows"
    sample += f", {n_frac:.4g} of the output rows of every contraction, per step (quantize included)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; distributions of the benchmark definition)",
            "config": {"workload": cfg["name"], "config_id": args.config, "M": cfg["M"]},
            "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, ws, rank, local):
    import quantized_q8_activation_gb300 as qk
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    qk.build()
    qk.lib()
    cfg = CONFIGS[args.config]
    wl = Workload(args.config, seed=0, copies=args.copies)
    stream = torch.cuda.Stream(device)
    C = wl.copies
    S = C * max(1, -(-args.graph_steps // C))        # steps per graph, a multiple of the copy count

    front_end = args.front_end

    def steps(n, start=0, pdl=True, front_end=front_end):
        for i in range(n):
            wl.step((start + i) % C, pdl=pdl, stream=stream, front_end=front_end)

    # warm-up (also settles per-kernel attributes before any capture)
    with torch.cuda.stream(stream):
        steps(max(args.warmup, 1))
    torch.cuda.synchronize()
    g_main = capture(lambda: steps(S), stream)
    rem = args.steps % S
    g_rem = capture(lambda: steps(rem), stream) if rem else None
    nrep = args.steps // S
    g_main.replay()                                     # one untimed replay of the graph itself
    torch.cuda.synchronize()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(nrep):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            e1.record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    ms = e0.elapsed_time(e1)
    ms = barrier_max(ms, ws, device)
    ms_step = ms / args.steps

    # the same step with the other activation paths, for reference
    front_end_ms = {}
    if cfg["kind"] == "gemv":
        for fe in ("fused", "unfused"):
            if fe == front_end:
                continue
            g_alt = capture(lambda: steps(S, front_end=fe), stream)
            g_alt.replay()
            torch.cuda.synchronize()
            reps = max(1, min(nrep, 50))
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a0.record(stream)
                for _ in range(reps):
                    g_alt.replay()
                a1.record(stream)
            torch.cuda.synchronize()
            front_end_ms[fe] = a0.elapsed_time(a1) / (reps * S)
            del g_alt
        front_end_ms[front_end] = ms_step

    # Per-kernel durations: each kernel type's launches of one step, S steps of them back to back
    # in a graph of their own (same launch configuration as the step: PDL, rotating weight copies),
    # timed with CUDA events on the launching stream.
    groups = {}
    for gemm in cfg["gemms"]:
        f = gemm_fused(front_end, cfg, gemm)
        groups.setdefault(wl.kernel_key(gemm, f), []).append((gemm, f))
    per_kernel = {}
    for key, gf in groups.items():
        gl = [g for g, _ in gf]
        gk = capture(lambda: [wl.launch(g, i % C, pdl=True, stream=stream, fused=f)
                              for i in range(S) for g, f in gf], stream)
        gk.replay()
        torch.cuda.synchronize()
        reps = max(1, min(nrep, 20))
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            k0.record(stream)
            for _ in range(reps):
                gk.replay()
            k1.record(stream)
        torch.cuda.synchronize()
        del gk
        n_launch = reps * S * len(gl)
        per_kernel[key] = {"ms": k0.elapsed_time(k1) / (reps * S),          # per step
                           "n": len(gl),                                     # calls per step
                           "avg_us": k0.elapsed_time(k1) / n_launch * 1e3,
                           "bytes": sum(N * (K // 256) * BYTES_PER_SB[q] for (_, q, N, K, _, _) in gl),
                           "ops": sum(2 * cfg["M"] * N * K for (_, _, N, K, _, _) in gl)}
    dom = max(per_kernel, key=lambda k: per_kernel[k]["ms"])
    dk = per_kernel[dom]
    hbm, bf16, peak_src = peaks()
    traffic = recorded_traffic(args.config, dom)

    if cfg["kind"] == "mmq":
        units = int_ops(cfg)
        value = units * ws / (ms_step * 1e-3) / 1e12
        unit = "TOPS"
        achieved = dk["ops"] / (dk["ms"] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                "frac": achieved / bf16, "traffic": traffic, "kernel": dom,
                "algorithmic_ops_per_launch": dk["ops"] / dk["n"],
                "peak_note": f"f16 tensor path: bf16 dense {peak_src} x nominal f16/bf16 ratio 1; "
                             "achieved counts the algorithmic 2*M*N*K integer ops (the kernel issues "
                             + ("two f16 MMAs per product (A_hi, A_lo against the exact sc*q) plus the "
                                "K/32-deep min-term contraction" if dom == "mmq_q4k" else
                                "three f16 MMAs per product for the hi/lo split") + "); a launch here is one "
                             "qk_mmq call, its prep kernel and its main kernel",
                "avg_launch_us": dk["avg_us"]}
    else:
        units = weight_bytes(cfg)
        value = units * ws / (ms_step * 1e-3) / 1e9
        unit = "GB/s"
        achieved = dk["bytes"] / (dk["ms"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic, "kernel": dom, "peak_note": f"hbm_gbs ({peak_src}, burst copy)",
                "algorithmic_bytes_per_launch": dk["bytes"] / dk["n"],
                "avg_launch_us": dk["avg_us"]}

    # end to end through the public API with host buffers (pinned), copies inside the timed region
    h2d = {s: torch.from_numpy(v).pin_memory() for s, v in wl.host_x.items()}
    h2r = {n: torch.from_numpy(v).pin_memory() for n, v in wl.host_r.items()}
    d2h = {n: torch.empty(tuple(t.shape), dtype=torch.float32).pin_memory() for n, t in wl.y.items()}
    h2d_bytes = sum(t.numel() * 4 for t in h2d.values()) + sum(t.numel() * 4 for t in h2r.values())
    d2h_bytes = sum(t.numel() * 4 for t in d2h.values())

    def e2e_step(i):
        for s, t in h2d.items():
            wl.x[s].copy_(t, non_blocking=True)
        for n, t in h2r.items():
            wl.r[n].copy_(t, non_blocking=True)
        wl.step(i % C, pdl=True, stream=stream, front_end=front_end)
        for n, t in d2h.items():
            t.copy_(wl.y[n], non_blocking=True)

    e2e_steps = min(args.steps, max(S, 200))
    g_e2e = capture(lambda: [e2e_step(i) for i in range(S)], stream)
    g_e2e.replay()
    torch.cuda.synchronize()
    reps = max(1, e2e_steps // S)
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g_e2e.replay()
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / (reps * S)
    e2e_s = barrier_max(e2e_s, ws, device)
    e2e_value = (units * ws / e2e_s / (1e12 if unit == "TOPS" else 1e9))

    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8",
            "data": "synthetic (seeded; distributions of the benchmark definition)",
            "config": {"workload": cfg["name"], "config_id": args.config, "M": cfg["M"],
                       "weight_bytes_per_step": weight_bytes(cfg), "int_ops_per_step": int_ops(cfg),
                       "l2": f"inputs larger than L2: {C} rotating weight copies, "
                             f"{C * weight_bytes(cfg) / 1e6:.0f} MB working set",
                       "graph_steps": S, "pdl": True, "parallelism": f"replicas x{ws}",
                       "front_end": front_end_desc(front_end, cfg)},
            "front_end_ms_per_step": front_end_ms or None,
            "hbm_frac": (value / ws) / hbm if unit == "GB/s" else None,
            "roofline": roof,
            # per entry point: its calls per step (an MMQ call is two kernels, prep and main), the
            # average call time and its share of the entry points' time
            "per_kernel": {k: {"calls_per_step": v["n"], "avg_us": v["avg_us"],
                               "share": v["ms"] / sum(x["ms"] for x in per_kernel.values())}
                           for k, v in per_kernel.items()},
            "clocks": clk.summary(),
            "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d_bytes,
                    "d2h_bytes_per_step": d2h_bytes, "ms_per_step": e2e_s * 1e3},
            "gpu_launches": wl.launches_per_step(front_end) * args.steps}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline((wl.host_w, wl.host_x, wl.host_r), cfg, budget_s=args.cpu_seconds,
                                            host_g=wl.host_g)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default per config: about a second of GPU work)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, choices=sorted(CONFIGS))
    ap.add_argument("--copies", type=int, default=None, help="weight copies rotated between steps")
    ap.add_argument("--graph-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: total host time the warm-up and timed steps are sized to")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--front-end", choices=["auto", "fused", "unfused"], default="auto",
                    help="decode activation path: q8_1 quantization inside each GEMV (fused) or a "
                         "quantize kernel before its consumers (unfused); auto = fused for activations "
                         "of at most 4096 values, unfused for larger ones")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = {0: 100000, 1: 40000, 2: 10000, 3: 8000, 4: 100, 5: 100, 6: 40000, 7: 40000, 8: 30000,
                      9: 40000, 10: 40000}[args.config]
    args.graph_steps = max(1, min(args.graph_steps, args.steps))
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank)
        else:
            run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
