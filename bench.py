#!/usr/bin/env python3
"""Benchmark of the k-quant x q8_1 contraction on GB300.

One "step" is one pass of the whole hot path over one batch of synthetic
input: q8_1 quantization of every distinct activation, then the GEMV (decode)
or MMQ (prefill) of every weight that reads it, residual adds fused.

Workloads (benchmark configurations; shapes of the named models, synthetic
data of the stated distributions):
  0  single Q4_K GEMV 4096 x 4096, M = 1
  1  Llama-3-8B decode layer, M = 1: QKV 6144x4096, attn-out 4096x4096 (+res),
     gate||up 28672x4096 (one q8_1 activation), down 4096x14336 (+res)   [headline]
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

Default run: config 1 is the headline line; configs 0, 2, 3 and 4 are timed
with the same --steps / --warmup and reported under "configs" in the same
JSON line, with the measured tensor-core peaks for the MMQ.  --config N times
only workload N.

Timing: W untimed warm-up steps, then exactly K steps replayed from CUDA
graphs (programmatic dependent launch between the kernels), bracketed by a
barrier and torch.cuda.synchronize().  The K steps are split into R >= 5
graph replays of S steps, each timed with its own CUDA events on the
launching stream; ms_per_step is the median replay per step, with the
spread and the all-K total beside it.  Weight copies rotate between steps so
the working set exceeds L2.  `--impl reference` times the CPU oracle on the
host cores instead.
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
    """Activation path of one GEMM: q8_1 quantization inside the contraction ("fused")
    or a quantize kernel before its consumers.  Decode: "auto" quantizes inside the GEMV
    when the activation is small (M*K <= 4096: one float4 or two per thread), where
    saving the extra kernel and dependency wins; larger activations use the quantize
    kernel, since the in-GEMV front end repeats the quantization in every CTA.  Prefill:
    the MMQ's prep kernel quantizes once per call, so every policy but "unfused" fuses.
    The decode chain fuses only attn-out, the one f32 activation it does not produce."""
    if cfg["kind"] == "chain":
        return gemm[0] == "attn_out"
    if cfg["kind"] == "mmq":
        return policy != "unfused"
    if cfg["kind"] != "gemv":
        return False
    if policy == "auto":
        return cfg["M"] * gemm[3] <= 4096
    return policy == "fused"                        # "unfused" and "batched" read q8_1


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, averaged over the
# kernel's launches in one step) from one ncu capture of the command in the named profile.
# Valid only while the kernel sources are the ones the counters were taken on.
TRAFFIC: dict = {
    (0, "gemv_q4k"): {"bytes_per_launch": 9464504, "digest": "196408130cfd657b",
                      "profile": "profiles/dram_traffic_per_launch.md"},
    (1, "gemv_q4k"): {"bytes_per_launch": 30709863, "digest": "196408130cfd657b",
                      "profile": "profiles/launches_llama3_8b_decode_layer.md"},
    (2, "gemv_q6k"): {"bytes_per_launch": 434436890, "digest": "196408130cfd657b",
                      "profile": "profiles/gemv_q6k_head_128256x4096.md"},
    (3, "gemv_q6k"): {"bytes_per_launch": 435223040, "digest": "196408130cfd657b",
                      "profile": "profiles/gemv_q6k_head_m4_128256x4096.md"},
    (4, "mmq_q4k_f32"): {"bytes_per_launch": 332174272, "digest": "7dc433405fca68ba",
                         "profile": "profiles/launches_qwen2_7b_prefill_mmq.md"},
}


def front_end_desc(front_end: str, cfg) -> str:
    if cfg["kind"] == "chain":
        return ("producers: qk_rmsnorm_q8_1 -> qkv; attn_out quantizes its f32 input inside the GEMV; "
                "qk_rmsnorm_q8_1 -> gate_up; qk_swiglu_q8_1 -> down")
    if cfg["kind"] == "mmq":
        return ("q8_1 quantization inside each MMQ call (qk_mmq_*_f32)" if front_end != "unfused"
                else "qk_quantize_q8_1 kernel per activation, then the q8_1 MMQ entry points")
    if cfg["kind"] != "gemv":
        return "qk_quantize_q8_1 kernel per activation"
    if front_end == "batched":
        return ("batched: one qk_quantize_q8_1 launch over all of the step's f32 activations (contiguous in "
                "the input buffer), then every GEMV reads q8_1")
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
    if front_end == "batched" and cfg["kind"] == "gemv":
        return 1 + len(cfg["gemms"])
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

def packed(shapes, device, align: int = 128):
    """One zero-filled float32 buffer holding a tensor of each shape (offsets aligned to `align`
    elements); returns the buffer, the views and the offsets."""
    offs, n = [], 0
    for sh in shapes:
        offs.append(n)
        n += -(-int(np.prod(sh)) // align) * align
    buf = torch.zeros(max(n, align), dtype=torch.float32, device=device)
    return buf, [buf[o:o + int(np.prod(sh))].view(*sh) for o, sh in zip(offs, shapes)], offs


class Workload:
    """Device buffers for one configuration: repacked weights (several copies),
    f32 activations and residuals, q8_1 buffers and outputs."""

    def __init__(self, cfg_id: int, seed: int = 0, copies: int | None = None, device="cuda", mmq_plane: bool = False):
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
        # inputs (f32 activations and residuals) and outputs live in one packed device buffer
        # each, so an end-to-end step moves them with one copy per direction
        chain = cfg["kind"] == "chain"
        x_specs = [(s, (M, K)) for s, K in slots(cfg) if s in cfg.get("inputs", [s])]
        r_specs = [(name, (M, N)) for (name, _, N, _, res, _) in cfg["gemms"] if res and not (chain and name == "down")]
        y_specs = [(name, (M, N)) for (name, _, N, _, _, _) in cfg["gemms"]]
        self._specs = (x_specs, r_specs, y_specs)
        self.host_x = {s: synth.activations(M, sh[1], seed=seed, tag=s) for s, sh in x_specs}
        self.host_r = {n: synth.residual(M, sh[1], seed=seed, tag=n) for n, sh in r_specs}
        self.host_g = {}
        if chain:
            self.host_g = chain_norm_weights(cfg, seed)
            self.g = {t: torch.from_numpy(v).to(device) for t, v in self.host_g.items()}
        self.banks = [self._make_bank(device)]
        self.use_bank(0)
        self.ws = None
        # Q4_K MMQ with load-time min-operand planes (built here, with the weights, outside any timing)
        self.plane = [dict() for _ in range(copies)]
        if cfg["kind"] == "mmq" and mmq_plane:
            for (name, q, N, K, _, _) in cfg["gemms"]:
                if q == "q4k":
                    for c in range(copies):
                        self.plane[c][name] = qk.q4k_min_plane(self.w[c][name], N, K)
        if cfg["kind"] == "mmq":
            need = max(qk.mmq_workspace_bytes(M, N, K) for (_, _, N, K, _, _) in cfg["gemms"])
            self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device) if need else None
        torch.cuda.synchronize()

    def _make_bank(self, device):
        """One set of step buffers: the packed f32 inputs (activations, then residuals), their
        q8_1 codes and scales packed the same way, and the packed outputs."""
        x_specs, r_specs, y_specs = self._specs
        M, qk = self.M, self.qk
        inbuf, views, offs = packed([sh for _, sh in x_specs + r_specs], device)
        b = {"inbuf": inbuf, "x": {s: v for (s, _), v in zip(x_specs, views[:len(x_specs)])},
             "r": {n: v for (n, _), v in zip(r_specs, views[len(x_specs):])}}
        # the activations come first: their q8_1 codes and scales are packed the same way, so one
        # quantize launch over the prefix quantizes every activation of the step (32-value blocks
        # never cross an activation, whose sizes and offsets are multiples of 128 values)
        b["x_prefix"] = n = offs[len(x_specs)] if r_specs else inbuf.numel()
        b["q8_codes"] = torch.empty(n, dtype=torch.int8, device=device)
        b["q8_scales"] = torch.empty((n // 32, 2), dtype=torch.float16, device=device)
        x_off = {s: o for (s, _), o in zip(x_specs, offs)}
        b["outbuf"], yv, _ = packed([sh for _, sh in y_specs], device)
        b["y"] = {n_: v for (n_, _), v in zip(y_specs, yv)}
        for s, v in self.host_x.items():
            b["x"][s].copy_(torch.from_numpy(v))
        for n_, v in self.host_r.items():
            b["r"][n_].copy_(torch.from_numpy(v))
        b["q8"] = {}
        for s, K in slots(self.cfg):
            if s in x_off:
                o = x_off[s]
                b["q8"][s] = (b["q8_codes"][o:o + M * K].view(M, K),
                              b["q8_scales"][o // 32:(o + M * K) // 32].view(M, K // 32, 2))
            else:
                b["q8"][s] = qk.empty_q8_1(M, K, device)
        if self.cfg["kind"] == "chain":
            b["r"]["down"] = b["y"]["attn_out"]     # down adds the residual stream h = attn-out's output
        return b

    def add_bank(self):
        """A second set of step buffers (pipelined end-to-end steps alternate between the two)."""
        if len(self.banks) < 2:
            self.banks.append(self._make_bank(self.inbuf.device))

    def use_bank(self, i: int):
        b = self.banks[i]
        self.inbuf, self.x, self.r, self.outbuf, self.y, self.q8 = b["inbuf"], b["x"], b["r"], b["outbuf"], b["y"], b["q8"]
        self.x_prefix, self.q8_codes, self.q8_scales = b["x_prefix"], b["q8_codes"], b["q8_scales"]

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
            if cfg["kind"] == "mmq" and fused:
                # the f32 activation quantized inside the call (the q8_1 buffers are not touched)
                plane = self.plane[copy].get(name)
                if q == "q4k":
                    qk.mmq_q4k_f32(self.w[copy][name], self.x[s], N, K, workspace=self.ws, plane=plane, **kw)
                else:
                    qk.mmq_q6k_f32(self.w[copy][name], self.x[s], N, K, workspace=self.ws, **kw)
            elif cfg["kind"] == "mmq":
                ws = self.ws
                plane = self.plane[copy].get(name)
                if plane is not None:
                    qk.mmq_q4k_plane(self.w[copy][name], plane, codes, scales, N, K, workspace=ws, **kw)
                else:
                    fn = qk.mmq_q4k if q == "q4k" else qk.mmq_q6k
                    fn(self.w[copy][name], codes, scales, N, K, workspace=ws, **kw)
            else:
                fn = {"q4k": qk.gemv_q4k, "q5k": qk.gemv_q5k, "q6k": qk.gemv_q6k, "q80": qk.gemv_q8_0,
                      "q2k": qk.gemv_q2k, "q3k": qk.gemv_q3k}[q]
                fn(self.w[copy][name], codes, scales, N, K, **kw)

    def step(self, copy: int, pdl: bool = True, stream=None, front_end: str = "batched"):
        """Enqueue one step on `stream`.  Each decode GEMM either quantizes its activation
        inside the GEMV (qk_gemv_*_f32) or reads the q8_1 codes of a quantize kernel that
        runs once per activation before its first consumer (see gemm_fused)."""
        qk, cfg = self.qk, self.cfg
        if cfg["kind"] == "chain":
            return self.chain_step(copy, pdl, stream)
        if front_end == "batched" and cfg["kind"] == "gemv":
            self.quantize_all(pdl, stream)
            for gemm in cfg["gemms"]:
                self.launch(gemm, copy, pdl=pdl, stream=stream, fused=False)
            return
        done = set()
        for gemm in cfg["gemms"]:
            s = gemm[5]
            fused = gemm_fused(front_end, cfg, gemm)
            if not fused and s not in done:
                codes, scales = self.q8[s]
                qk.quantize_q8_1(self.x[s], codes, scales, pdl=pdl, stream=stream)
                done.add(s)
            self.launch(gemm, copy, pdl=pdl, stream=stream, fused=fused)

    def quantize_all(self, pdl: bool, stream):
        """One qk_quantize_q8_1 launch over every f32 activation of the step (the packed prefix)."""
        n = self.x_prefix
        self.qk.quantize_q8_1(self.inbuf[:n].view(1, n), self.q8_codes.view(1, n),
                              self.q8_scales.view(1, n // 32, 2), pdl=pdl, stream=stream)

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
            return ("mmq_q4k" if q == "q4k" else "mmq_q6k") + ("_f32" if fused else "")
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


def cpu_baseline(wl_host, cfg, budget_s: float = 12.0, host_g=None, threads=None):
    """Time the oracle as it stands on the host cores (all of them, or `threads`); bounded sample."""
    threads = threads or os.cpu_count() or 1
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


class StepGraphs:
    """The timed region of K steps, step i using weight copy i % C.
    K <= S (one graph holds the region): the region is one CUDA graph of K steps, so programmatic
    dependent launch links every step, and it is replayed `regions` times, each replay timed.
    K > S: the region is R = K // S graphs of S steps (R >= 5 by the choice of S) plus a remainder
    graph, each full replay timed.  Graphs with the same copy sequence are captured once."""

    def __init__(self, step_fn, K: int, S: int, C: int, stream, regions: int = 5):
        if K <= S:
            S = K
        self.S = S
        self.R, self.rem = (regions, 0) if K == S else (K // S, K % S)
        cache = {}

        def graph(off, n):
            key = (off, n)
            if key not in cache:
                cache[key] = capture(lambda: [step_fn((off + i) % C) for i in range(n)], stream)
            return cache[key]

        self.plan = [graph(0 if K == S else (r * S) % C, S) for r in range(self.R)]
        self.tail = graph((self.R * S) % C, self.rem) if self.rem else None
        self.graphs = list(cache.values())

    def warm(self):
        for g in self.graphs:
            g.replay()
        torch.cuda.synchronize()

    def run_timed(self, stream):
        """Replay the region (K steps, or `regions` times K steps when one graph holds it), each
        full replay between its own pair of events; returns the per-step milliseconds of each
        full replay and the total milliseconds."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(self.R + 2)]
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for r, g in enumerate(self.plan):
                g.replay()
                ev[r + 1].record(stream)
            if self.tail is not None:
                self.tail.replay()
            ev[-1].record(stream)
        torch.cuda.synchronize()
        per = [ev[r].elapsed_time(ev[r + 1]) / self.S for r in range(self.R)]
        return per, ev[0].elapsed_time(ev[-1])


def steps_per_replay(K: int, graph_steps: int) -> int:
    """Steps per graph: all K when one graph of at most graph_steps holds them (the region is then
    replayed five times), else at most graph_steps and small enough for five replays or more."""
    return K if K <= graph_steps else max(1, min(graph_steps, K // 5))


def time_graphs(step_fn, K, S, C, stream):
    sg = StepGraphs(step_fn, K, S, C, stream)
    sg.warm()
    per, total = sg.run_timed(stream)
    del sg
    return per, total


def kernel_groups(wl, front_end):
    """The step's launches grouped by kernel family (the quantize kernels as their own group), in
    step order: {key: [(kind, gemm or slot, fused)]}."""
    cfg, groups, done = wl.cfg, {}, set()
    if front_end == "batched" and cfg["kind"] == "gemv":
        groups["quantize_q8_1"] = [("quantize_all", None, False)]
        for gemm in cfg["gemms"]:
            groups.setdefault(wl.kernel_key(gemm, False), []).append(("gemm", gemm, False))
        return groups
    for gemm in cfg["gemms"]:
        f = gemm_fused(front_end, cfg, gemm)
        if not f and gemm[5] not in done and cfg["kind"] != "chain":     # the chain's producers quantize
            groups.setdefault("quantize_q8_1", []).append(("quantize", gemm[5], False))
            done.add(gemm[5])
        groups.setdefault(wl.kernel_key(gemm, f), []).append(("gemm", gemm, f))
    return groups


def measure_config(cfg_id, args, stream, ws, device, peaks_meas=None, headline=False):
    """Time one workload: the K-step region (median of replays), each kernel family on its own,
    the end-to-end path with host buffers, and the roofline of the dominant kernel."""
    import quantized_q8_activation_gb300 as qk
    cfg = CONFIGS[cfg_id]
    front_end = args.front_end
    wl = Workload(cfg_id, seed=0, copies=args.copies, mmq_plane=args.mmq_min_operands == "plane")
    C, K = wl.copies, args.steps
    S = steps_per_replay(K, args.graph_steps)
    units = int_ops(cfg) if cfg["kind"] == "mmq" else weight_bytes(cfg)
    unit, scale = ("TOPS", 1e12) if cfg["kind"] == "mmq" else ("GB/s", 1e9)

    def step(copy, fe=front_end):
        wl.step(copy, pdl=True, stream=stream, front_end=fe)

    # warm-up (also settles per-kernel attributes before any capture)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i % C)
    torch.cuda.synchronize()

    sg = StepGraphs(step, K, S, C, stream)
    sg.warm()
    barrier(ws)
    torch.cuda.synchronize()
    per, total_ms = sg.run_timed(stream)
    barrier(ws)
    del sg
    med = statistics.median(per)
    ms_step = barrier_max(med, ws, device)
    total_ms = barrier_max(total_ms, ws, device)

    out = {"workload": cfg["name"], "config_id": cfg_id, "M": cfg["M"],
           "value": units * ws / (ms_step * 1e-3) / scale, "unit": unit, "ms_per_step": ms_step,
           "timing": {"replays": len(per), "steps_per_replay": S,
                      "how": (f"the {K}-step region as one graph, replayed {len(per)} times, each replay timed"
                              if S == K else f"{K} steps as {len(per)} timed replays of {S}-step graphs"),
                      "ms_per_step_median": med, "ms_per_step_min": min(per), "ms_per_step_max": max(per),
                      "ms_per_step_all_replays": total_ms / (S * len(per) + (K % S if S < K else 0)),
                      "weight_copies": C},
           "tokens_per_s": cfg["M"] * ws / (ms_step * 1e-3),
           "weight_bytes_per_step": weight_bytes(cfg), "int_ops_per_step": int_ops(cfg),
           "front_end": front_end_desc(front_end, cfg),
           "gpu_launches": wl.launches_per_step(front_end) * K}
    if unit == "GB/s":
        out["hbm_frac"] = (out["value"] / ws) / peaks()[0]
    if cfg["kind"] == "mmq":
        out["mmq"] = {"tile_width": "chosen per GEMM by the library (128, 192 or 256)", "split_k": "off",
                      "min_operands": "load-time plane (qk_q4k_min_plane)" if args.mmq_min_operands == "plane"
                      else "built in every tile from the 6-bit fields"}

    # the same step with the other decode activation paths, for reference
    if headline and cfg["kind"] == "gemv":
        fe_ms = {front_end: ms_step}
        for fe in ("fused", "unfused", "auto", "batched"):
            if fe != front_end:
                p2, _ = time_graphs(lambda c, fe=fe: step(c, fe), K, S, C, stream)
                fe_ms[fe] = statistics.median(p2)
        out["front_end_ms_per_step"] = fe_ms

    # Per kernel family: the step's launches of that family only, S steps of them back to back in
    # graphs of their own (same launch configuration: PDL, rotating weight copies), timed with CUDA
    # events on the launching stream; median over the replays.
    per_kernel = {}
    for key, items in kernel_groups(wl, front_end).items():
        def launches(copy, items=items):
            for kind, what, f in items:
                if kind == "quantize_all":
                    wl.quantize_all(True, stream)
                elif kind == "quantize":
                    codes, scales = wl.q8[what]
                    qk.quantize_q8_1(wl.x[what], codes, scales, pdl=True, stream=stream)
                else:
                    wl.launch(what, copy, pdl=True, stream=stream, fused=f)
        p2, _ = time_graphs(launches, K, S, C, stream)
        kms = statistics.median(p2)
        gl = [w for kind, w, _ in items if kind == "gemm"]
        nb = sum(N * (K_ // 256) * BYTES_PER_SB[q] for (_, q, N, K_, _, _) in gl)
        nops = sum(2 * cfg["M"] * N * K_ for (_, _, N, K_, _, _) in gl)
        act = sum(cfg["M"] * dict(slots(cfg))[w] * 4 for kind, w, _ in items if kind == "quantize")
        act += sum(wl.x_prefix * 4 for kind, _, _ in items if kind == "quantize_all")
        per_kernel[key] = {"calls_per_step": len(items), "ms_per_step": kms, "avg_us": kms / len(items) * 1e3,
                           "weight_bytes": nb, "ops": nops, "activation_bytes_in": act}
    tot = sum(v["ms_per_step"] for v in per_kernel.values()) or 1.0
    for v in per_kernel.values():
        v["share"] = v["ms_per_step"] / tot
        if v["weight_bytes"]:
            v["weight_gbs"] = v["weight_bytes"] / (v["ms_per_step"] * 1e-3) / 1e9
        if v["ops"] and cfg["kind"] == "mmq":
            v["tops"] = v["ops"] / (v["ms_per_step"] * 1e-3) / 1e12
        if v["activation_bytes_in"]:
            v["activation_gbs"] = v["activation_bytes_in"] / (v["ms_per_step"] * 1e-3) / 1e9
    out["per_kernel"] = per_kernel
    # per GEMM: its contraction call alone, in the same launch configuration
    per_gemm = {}
    for gemm in cfg["gemms"]:
        f = gemm_fused(front_end, cfg, gemm)
        p2, _ = time_graphs(lambda copy, g=gemm, f=f: wl.launch(g, copy, pdl=True, stream=stream, fused=f),
                            K, S, C, stream)
        us = statistics.median(p2) * 1e3
        name, q, N, K_, _, _ = gemm
        e = {"us": us, "kernel": wl.kernel_key(gemm, f)}
        if cfg["kind"] == "mmq":
            e["tops"] = 2 * cfg["M"] * N * K_ / (us * 1e-6) / 1e12
        else:
            e["weight_gbs"] = N * (K_ // 256) * BYTES_PER_SB[q] / (us * 1e-6) / 1e9
        per_gemm[name] = e
    out["per_gemm"] = per_gemm
    contraction = {k: v for k, v in per_kernel.items() if k != "quantize_q8_1"}
    if contraction:
        dom = max(contraction, key=lambda k: contraction[k]["ms_per_step"])
        out["roofline"] = roofline(cfg, cfg_id, dom, contraction[dom], peaks_meas)

    out["e2e"] = measure_e2e(wl, step, K, S, C, stream, ws, device, units, scale, unit)
    res = (wl.host_w, wl.host_x, wl.host_r, wl.host_g)
    del wl
    torch.cuda.empty_cache()
    return out, res


def roofline(cfg, cfg_id, dom, dk, peaks_meas):
    hbm, bf16, peak_src = peaks()
    traffic = recorded_traffic(cfg_id, dom)
    n = dk["calls_per_step"]
    if cfg["kind"] == "mmq":
        achieved = dk["ops"] / (dk["ms_per_step"] * 1e-3) / 1e12
        # f16 tensor MMAs the kernel issues per algorithmic integer product: two (A_hi, A_lo against the exact
        # sc*q) plus the min term's K/32-deep contraction (3 MMAs per 16 sub-blocks, ~4.7 % more) for Q4_K;
        # three (hi/lo splits) for Q6_K
        mma_per_product = (2.0 + 3.0 / 64.0) if dom.startswith("mmq_q4k") else 3.0
        r = {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s", "frac": achieved / bf16,
             "traffic": traffic, "kernel": dom, "algorithmic_ops_per_launch": dk["ops"] / n,
             "avg_launch_us": dk["avg_us"],
             "peak_note": f"bf16 dense {peak_src} (MEASURED_PEAKS.json) x nominal f16/bf16 ratio 1; achieved counts "
                          "the algorithmic 2*M*N*K integer ops; a launch is one qk_mmq call (its prep and main kernel)",
             "f16_mma_per_integer_product": mma_per_product}
        if peaks_meas:
            f16p, s8p = peaks_meas.get("tcgen05_f16_tflops"), peaks_meas.get("mma_sync_s8_tops")
            if f16p:
                r["f16_tcgen05_peak"] = f16p
                r["frac_of_f16_tcgen05_peak"] = achieved / f16p
                r["issued_mma_utilisation"] = achieved * mma_per_product / f16p
            if s8p:
                r["int8_mma_sync_peak"] = s8p
                r["ratio_to_int8_mma_sync_peak"] = achieved / s8p
        return r
    achieved = dk["weight_bytes"] / (dk["ms_per_step"] * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": traffic, "kernel": dom, "peak_note": f"hbm_gbs ({peak_src}, burst copy)",
            "algorithmic_bytes_per_launch": dk["weight_bytes"] / n, "avg_launch_us": dk["avg_us"]}


def measure_e2e(wl, step, K, S, C, stream, ws, device, units, scale, unit):
    """The same metric through the public API with host buffers: every step copies its f32
    activations and residuals in from pinned host memory (one copy of the packed input block)
    and its outputs back out (one copy of the packed output block), inside the timed region.
    The steps alternate between two sets of device buffers, and the copies run on their own
    streams: step i's inputs arrive while step i - 1 computes, and its outputs leave while
    step i + 1 computes (a bank's inputs are rewritten only after the step two before has
    finished with them, and its outputs only after their copy out has finished)."""
    wl.add_bank()
    wl.use_bank(0)
    host_in = torch.empty(wl.inbuf.numel(), dtype=torch.float32).pin_memory()
    host_in.copy_(wl.inbuf.cpu())                  # same layout as the device blocks
    host_out = torch.empty(wl.outbuf.numel(), dtype=torch.float32).pin_memory()
    h2d, d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    Se = S if S % 2 == 0 else S + 1                # an even number of steps per graph: banks alternate

    def run(n, start=0):
        fork = torch.cuda.Event()
        fork.record(stream)
        h2d.wait_event(fork)
        d2h.wait_event(fork)
        done_c, done_out = [None, None], [None, None]
        for i in range(n):
            bk = i % 2
            wl.use_bank(bk)
            with torch.cuda.stream(h2d):
                if done_c[bk] is not None:
                    h2d.wait_event(done_c[bk])
                wl.inbuf.copy_(host_in, non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(h2d)
            stream.wait_event(e_in)
            if done_out[bk] is not None:
                stream.wait_event(done_out[bk])
            with torch.cuda.stream(stream):
                step((start + i) % C)
            e_c = torch.cuda.Event()
            e_c.record(stream)
            done_c[bk] = e_c
            with torch.cuda.stream(d2h):
                d2h.wait_event(e_c)
                host_out.copy_(wl.outbuf, non_blocking=True)
                e_out = torch.cuda.Event()
                e_out.record(d2h)
            done_out[bk] = e_out
        for e in done_out + done_c:                 # join the side streams back
            if e is not None:
                stream.wait_event(e)
        wl.use_bank(0)

    R = max(5, -(-K // Se))
    g = capture(lambda: run(Se), stream)
    g.replay()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(R + 1)]
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for r in range(R):
            g.replay()
            ev[r + 1].record(stream)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) * 1e3
    per = [ev[r].elapsed_time(ev[r + 1]) / Se for r in range(R)]
    del g
    ms = barrier_max(statistics.median(per), ws, device)
    return {"value": units * ws / (ms * 1e-3) / scale, "unit": unit,
            "h2d_bytes_per_step": wl.inbuf.numel() * 4, "d2h_bytes_per_step": wl.outbuf.numel() * 4,
            "ms_per_step": ms, "ms_per_step_wall": wall / (R * Se), "copies_per_step": 2,
            "how": f"{R} timed replays of a graph of {Se} steps; copies in and out on their own streams, "
                   "overlapping the neighbouring steps' compute (two alternating sets of device buffers)"}


def measure_peaks():
    """The two tensor-core ceilings of the prefill MMQ, measured on this device (include/qk_peak.h)."""
    import quantized_q8_activation_gb300 as qk
    f16, _ = qk.peak_tcgen05_f16(iters=4096, reps=10)
    s8, _ = qk.peak_mma_s8(iters=20000, reps=5)
    return {"tcgen05_f16_tflops": f16, "mma_sync_s8_tops": s8,
            "how": "own micro-benchmarks (include/qk_peak.h): tcgen05.mma kind::f16 128x256x16 back to back from one "
                   "thread per SM, and mma.sync m16n8k32 s8 with 8 chains per warp, 16 warps per SM; CUDA events"}


def run_ours(args, ws, rank, local):
    import quantized_q8_activation_gb300 as qk
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    qk.build()
    qk.lib()
    stream = torch.cuda.Stream(device)
    head = args.config if args.config is not None else 1
    extra = [] if args.config is not None else [0, 2, 3, 4]
    ids = [head] + extra
    need_peaks = any(CONFIGS[c]["kind"] == "mmq" for c in ids)
    with ClockSampler(local) as clk:
        peaks_meas = measure_peaks() if need_peaks else None
        results, hosts = {}, {}
        for c in ids:
            steps0 = args.steps
            if args.steps is None:
                args.steps = DEFAULT_STEPS[c]
            results[c], host = measure_config(c, args, stream, ws, device, peaks_meas, headline=(c == head))
            if c == head or CONFIGS[c]["kind"] == "mmq":          # the workloads the oracle baseline times
                hosts[c] = host
            args.steps = steps0
    h = results[head]
    cfg = CONFIGS[head]
    line = {"metric": METRIC, "value": h["value"], "unit": h["unit"], "n_gpus": ws,
            "steps": args.steps if args.steps is not None else DEFAULT_STEPS[head], "warmup": args.warmup,
            "ms_per_step": h["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8", "data": "synthetic (seeded; distributions of the benchmark definition)",
            "config": {"workload": cfg["name"], "config_id": head, "M": cfg["M"],
                       "weight_bytes_per_step": weight_bytes(cfg), "int_ops_per_step": int_ops(cfg),
                       "l2": f"inputs larger than L2: {h['timing']['weight_copies']} rotating weight copies, "
                             f"{h['timing']['weight_copies'] * weight_bytes(cfg) / 1e6:.0f} MB working set",
                       "pdl": True, "parallelism": f"replicas x{ws}", "front_end": h["front_end"]},
            "timing": h["timing"], "tokens_per_s": h["tokens_per_s"]}
    for k in ("front_end_ms_per_step", "hbm_frac", "roofline", "per_kernel", "per_gemm"):
        if k in h:
            line[k] = h[k]
    line["clocks"] = clk.summary()
    line["e2e"] = h["e2e"]
    line["gpu_launches"] = h["gpu_launches"]
    if peaks_meas:
        line["tensor_peaks"] = peaks_meas
    if extra:
        line["configs"] = {str(c): results[c] for c in extra}
    if rank == 0 and not args.no_cpu_baseline:
        hw, hx, hr, hg = hosts[head]
        line["cpu_baseline"] = cpu_baseline((hw, hx, hr), cfg, budget_s=args.cpu_seconds, host_g=hg)
        line["cpu_baseline_1thread"] = cpu_baseline((hw, hx, hr), cfg, budget_s=args.cpu_seconds, host_g=hg,
                                                    threads=1)
        for c in extra:
            if CONFIGS[c]["kind"] == "mmq":
                hw, hx, hr, hg = hosts[c]
                line["configs"][str(c)]["cpu_baseline"] = cpu_baseline((hw, hx, hr), CONFIGS[c],
                                                                       budget_s=args.cpu_seconds / 2, host_g=hg)
    if rank == 0:
        print(json.dumps(line), flush=True)


DEFAULT_STEPS = {0: 100000, 1: 40000, 2: 10000, 3: 8000, 4: 100, 5: 100, 6: 40000, 7: 40000, 8: 30000,
                 9: 40000, 10: 40000}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps of every workload (default per workload: about a second of GPU work)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=None, choices=sorted(CONFIGS),
                    help="time only this workload (default: config 1 as the headline, with configs 0, 2, 3 "
                         "and 4 under 'configs')")
    ap.add_argument("--copies", type=int, default=None, help="weight copies rotated between steps")
    ap.add_argument("--graph-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: total host time the warm-up and timed steps are sized to")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mmq-min-operands", choices=["plane", "tile"], default="plane",
                    help="prefill Q4_K MMQ: read the min-term operands from load-time planes built with the weights "
                         "(qk_q4k_min_plane, default; measured 1.8 %% faster per step) or build them from the 6-bit "
                         "fields in every tile")
    ap.add_argument("--front-end", choices=["batched", "auto", "fused", "unfused"], default="batched",
                    help="decode activation path: one quantize kernel over all of the step's f32 "
                         "activations, then q8_1 GEMVs (batched, default); q8_1 quantization inside each "
                         "GEMV (fused); a quantize kernel per activation before its consumers (unfused); "
                         "auto = fused for activations of at most 4096 values, unfused for larger ones")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps is not None and args.steps < 1:
        ap.error("--steps must be >= 1")
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    try:
        if args.impl == "reference":
            if args.config is None:
                args.config = 1
            if args.steps is None:
                args.steps = DEFAULT_STEPS[args.config]
            run_reference(args, ws, rank)
        else:
            run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
