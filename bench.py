#!/usr/bin/env python
"""Benchmark of the FP8 linear layer on GB300: block quantization + block-scaled
FP8 GEMM, reported as quant+GEMM TFLOP/s.

Default workload (the JSON line the contract asks for): the Llama-3.1-8B-shaped
fprop linears (M = 8192 tokens; QKV 4096->6144, O 4096->4096, gate+up
4096->28672, down 14336->4096; X per 1x128, W per 128x128, E4M3, fp32 scales,
bf16 out).  One step = for each linear: quantize X (1x128), re-quantize W
(128x128, the weights change every optimizer step), GEMM -> Y.

Other workloads (--workload): llama2-7b-fprop (pow2 scales, M=4096),
llama3.1-8b-fprop-mxfp8 (the same linears in MXFP8: 1x32 blocks, E8M0 scales),
llama3.1-8b-mlp-bwd (per-tensor delayed E5M2 dY, dgrad + wgrad on transposed
operands), llama3.1-8b-mlp-bwd-blockwise (the same backward under the block
recipe: row-wise and column-wise transposed 1x128 copies of dY and X),
qwen3-30b-a3b-moe (grouped expert GEMMs), llama3.1-8b-mlp-fused and
qwen3-30b-a3b-moe-fused (gate/up product with a SwiGLU + FP8-quantizing
epilogue feeding the down product directly), llama3.1-8b-attn-fp8 (causal
prefill attention over an FP8 KV cache, both products on FP8 tensor cores).

Inputs are synthetic (seeded), resident in HBM; every step streams more than
the 129 MB L2.

  python bench.py [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
Under torchrun (--gpus N) every rank runs the same workload on its own GPU
(independent replicas, weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time
from collections import defaultdict

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_scaled_gemm_quantize_gb300 import inputs as W_  # noqa: E402

METRIC = "block-scaled FP8 linear TFLOPS (quant+GEMM) and % of GB300 dense FP8 peak"
FP8_OVER_BF16 = 2.0      # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)
FLUSH_BYTES = 256 << 20  # written between timed steps: twice the 129 MB L2
KERNEL_SOURCES = ("block_scaled_gemm_quantize_gb300/csrc/gemm.cu",
                  "block_scaled_gemm_quantize_gb300/csrc/gemm_kernels.h",
                  "block_scaled_gemm_quantize_gb300/csrc/ptx_sm100.cuh",
                  "block_scaled_gemm_quantize_gb300/csrc/fp8_math.cuh")
# DRAM read+write bytes per GEMM launch (ncu dram__bytes_read.sum + dram__bytes_write.sum), per
# workload and linear, with the digest of the GEMM sources the counters were taken on.  The
# bench reports them only while the sources still have that digest (else traffic is null).
GEMM_TRAFFIC = {"sources_sha256": "1eba056e8de25b60",
                "bytes": {"llama3.1-8b-fprop": {"qkv": 134.14e6, "o": 80.01e6, "gate_up": 936.29e6,
                                                "down": 498.40e6}}}


def kernel_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


def reduce_max(v: float, device) -> float:
    """MAX of a host number over the ranks of the default process group (the
    contract's max-over-ranks timing); identity on one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dominant_kernel(wl):
    """Name of the kernel the roofline object describes (the workload's
    products): the attention kernel, the block-scaled (MX) GEMM for power-of-two
    or 1x32 scales on K-major operands, else the promotion GEMM."""
    if isinstance(wl, Attn):
        return "k_fp8_attn_fwd"
    if getattr(wl, "mx", False) or (isinstance(wl, (Fprop, FusedMlp)) and wl.mode == wl.fp8.SCALE_POW2):
        return "k_fp8_gemm_mx"
    return "k_fp8_gemm"


class Clocks:
    """nvidia-smi sampler running while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev: int):
        self.dev, self.rows, self.proc = dev, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in self.rows if num(r[0])]
        mx = [num(r[1]) for r in self.rows if num(r[1])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i] == "Active"})
        pw = [num(r[2]) for r in self.rows if num(r[2])]
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows),
                "power_w_max": max(pw) if pw else None}


class Rec:
    """Per-phase CUDA events on the launching (current) stream, kept per step."""

    def __init__(self):
        import torch
        self.torch, self.ev, self.step = torch, [], 0

    def __call__(self, kind, fn):
        e0 = self.torch.cuda.Event(enable_timing=True)
        e1 = self.torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        self.ev.append((self.step, kind, e0, e1))

    def medians(self):
        """Per phase: the median over steps of the phase's time in a step (ms)."""
        per = defaultdict(lambda: defaultdict(float))
        for step, kind, e0, e1 in self.ev:
            per[kind][step] += e0.elapsed_time(e1)
        return {k: float(np.median(list(v.values()))) for k, v in per.items()}


def _run(rec, kind, fn):
    if rec is None:
        fn()
    else:
        rec(kind, fn)


def _randn(g, shape, device, std=1.0):
    import torch
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _activations(g, M, K, device):
    """N(0,1) with round(1% of K) outlier channels x20 (bf16)."""
    import torch
    x = _randn(g, (M, K), device)
    cols = torch.randperm(K, generator=g, device=device)[: int(round(0.01 * K))]
    x[:, cols] *= 20.0
    return x.to(torch.bfloat16)


# ------------------------------------------------------------- workloads
class Fprop:
    """quant X (1x128) + quant W (128x128) + GEMM for each linear."""

    def __init__(self, cfg, fp8, device, seed=0, only=None):
        import torch
        self.cfg, self.fp8 = cfg, fp8
        self.mx = cfg["scale_mode"] == "mx"
        self.mode = fp8.SCALE_POW2 if cfg["scale_mode"] in ("pow2", "mx") else fp8.SCALE_FP32
        M = self.M = cfg["M"]
        g = torch.Generator(device=device)
        self.items = []
        for i, (name, N, K) in enumerate(cfg["linears"]):
            if only and name != only:
                continue
            g.manual_seed(seed * 1000 + i)
            x = _activations(g, M, K, device)
            w = (_randn(g, (N, K), device, 0.02)).to(torch.bfloat16)
            it = dict(name=name, N=N, K=K, x=x, w=w,
                      qx=torch.empty((M, K), dtype=torch.uint8, device=device),
                      qw=torch.empty((N, K), dtype=torch.uint8, device=device),
                      y=torch.empty((M, N), dtype=torch.bfloat16, device=device))
            if self.mx:   # MXFP8: E8M0 codes, one per 32 elements along K, both operands
                it["sx"] = torch.empty((K // 128, M, 4), dtype=torch.uint8, device=device)
                it["sw"] = torch.empty((K // 128, N, 4), dtype=torch.uint8, device=device)
                it["A"] = fp8.operand(it["qx"], it["sx"], fp8.E4M3, fp8.GRAN_1x32)
                it["B"] = fp8.operand(it["qw"], it["sw"], fp8.E4M3, fp8.GRAN_1x32)
            else:
                it["sx"] = torch.empty((K // 128, M), dtype=torch.float32, device=device)
                it["sw"] = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=device)
                it["A"] = fp8.operand(it["qx"], it["sx"], fp8.E4M3, fp8.GRAN_1x128)
                it["B"] = fp8.operand(it["qw"], it["sw"], fp8.E4M3, fp8.GRAN_128x128)
            self.items.append(it)
        if self.mx:
            self.units = [(it["name"], 2.0 * M * it["N"] * it["K"],
                           (M + it["N"]) * it["K"] * 3 + (M + it["N"]) * (it["K"] // 32))
                          for it in self.items]
        else:
            self.units = [(it["name"], 2.0 * M * it["N"] * it["K"],
                           M * it["K"] * 3 + 4 * M * (it["K"] // 128) + it["N"] * it["K"] * 3
                           + 4 * ((it["N"] + 127) // 128) * (it["K"] // 128)) for it in self.items]
        self.flops = sum(u[1] for u in self.units)
        self.launches = 3 * len(self.items)   # X and W quantization, GEMM
        self.config = self.static_config(cfg, only)

    @staticmethod
    def static_config(cfg, only=None):
        """The workload's config object (shared by both arms of the bench)."""
        return {"workload": cfg["name"] + (f" ({only} only)" if only else ""), "M": cfg["M"],
                "linears": [[n, N, K] for n, N, K in cfg["linears"] if not only or n == only],
                "scales": ("MXFP8: E8M0 per 1x32 (X and W)" if cfg["scale_mode"] == "mx"
                           else f"{cfg['scale_mode']} 1x128 (X) / 128x128 (W)"), "out": "bf16"}

    def step(self, rec=None):
        fp8, M, mode = self.fp8, self.M, self.mode
        for it in self.items:
            if self.mx:
                _run(rec, "quant:" + it["name"], lambda it=it: (
                    fp8.fp8_quantize_mx(it["x"], fp8.E4M3, q=it["qx"], scales=it["sx"]),
                    fp8.fp8_quantize_mx(it["w"], fp8.E4M3, q=it["qw"], scales=it["sw"])))
            else:   # X (1x128) and W (128x128) in one launch
                _run(rec, "quant:" + it["name"], lambda it=it: fp8.fp8_quantize_linear(
                    it["x"], it["w"], fp8.E4M3, mode, qx=it["qx"], sx=it["sx"], qw=it["qw"], sw=it["sw"]))
            _run(rec, "gemm:" + it["name"], lambda it=it: fp8.fp8_block_gemm(
                it["A"], it["B"], M, it["N"], it["K"], fp8.OUT_BF16, mode, y=it["y"]))

    def host_io(self):
        return [it["x"] for it in self.items] + [it["w"] for it in self.items], [it["y"] for it in self.items]

    def e2e_units(self):
        """Per linear: (device inputs, device outputs, the linear's share of a step)."""
        fp8, M, mode = self.fp8, self.M, self.mode

        def unit(it):
            if self.mx:
                fp8.fp8_quantize_mx(it["x"], fp8.E4M3, q=it["qx"], scales=it["sx"])
                fp8.fp8_quantize_mx(it["w"], fp8.E4M3, q=it["qw"], scales=it["sw"])
            else:
                fp8.fp8_quantize_linear(it["x"], it["w"], fp8.E4M3, mode, qx=it["qx"], sx=it["sx"], qw=it["qw"],
                                        sw=it["sw"])
            fp8.fp8_block_gemm(it["A"], it["B"], M, it["N"], it["K"], fp8.OUT_BF16, mode, y=it["y"])

        return [([it["x"], it["w"]], [it["y"]], lambda it=it: unit(it)) for it in self.items]


class MlpBwd:
    """Backward of the Llama-3.1-8B MLP under the hybrid delayed recipe: per
    linear, dY (E5M2, per-tensor delayed) is quantized with the scale in use,
    dgrad dX = dY W (W stored transposed for the product) and wgrad
    dW = dY^T X (dY, X transposed) run with per-tensor scales, then the amax
    history of dY advances.  X and W are E4M3 per-tensor delayed (quantized
    once, as the forward pass leaves them)."""

    def __init__(self, cfg, fp8, device, seed=0, only=None):
        import torch
        self.fp8, self.M = fp8, cfg["M"]
        M = self.M
        g = torch.Generator(device=device)
        self.items = []
        for i, (name, n_out, k_in) in enumerate(cfg["linears"]):
            if only and name != only:
                continue
            g.manual_seed(seed * 1000 + 100 + i)
            # Student-t(nu) = N(0,1) / sqrt(chi2(nu)/nu), from the seeded generator
            z = _randn(g, (M, n_out), device)
            chi = sum(_randn(g, (M, n_out), device) ** 2 for _ in range(int(cfg["dy_nu"])))
            dy = (z / torch.sqrt(chi / cfg["dy_nu"]) * cfg["dy_scale"]).to(torch.bfloat16)
            del z, chi
            x = _activations(g, M, k_in, device)
            w = _randn(g, (n_out, k_in), device, 0.02).to(torch.bfloat16)
            st_dy = fp8.DelayedScaling(cfg["history_len"], fp8.E5M2, cfg["margin"], device=device)
            st_x = fp8.DelayedScaling(cfg["history_len"], fp8.E4M3, cfg["margin"], device=device)
            st_w = fp8.DelayedScaling(cfg["history_len"], fp8.E4M3, cfg["margin"], device=device)
            qx = st_x.quantize(x, update=True)   # one step gives X and W a measured scale
            qw = st_w.quantize(w, update=True)
            qx = st_x.quantize(x, q=qx, update=False)
            qw = st_w.quantize(w, q=qw, update=False)
            it = dict(name=name, n_out=n_out, k_in=k_in, dy=dy, st_dy=st_dy,
                      qdy=torch.empty((M, n_out), dtype=torch.uint8, device=device), qx=qx, qw=qw,
                      dx=torch.empty((M, k_in), dtype=torch.bfloat16, device=device),
                      dw=torch.empty((n_out, k_in), dtype=torch.float32, device=device))
            E4, E5, T = fp8.E4M3, fp8.E5M2, fp8.GRAN_TENSOR
            it["A_dg"] = fp8.operand(it["qdy"], st_dy.scale, E5, T)                   # [M][n_out]
            it["B_dg"] = fp8.operand(qw, st_w.scale, E4, T, transposed=True)          # W^T
            it["A_wg"] = fp8.operand(it["qdy"], st_dy.scale, E5, T, transposed=True)  # dY^T
            it["B_wg"] = fp8.operand(qx, st_x.scale, E4, T, transposed=True)          # X^T
            self.items.append(it)
        self.units = []
        for it in self.items:
            f = 2.0 * M * it["n_out"] * it["k_in"]
            self.units += [(it["name"] + ".dgrad", f, 0), (it["name"] + ".wgrad", f, 0)]
        self.quant_bytes = sum(3 * M * it["n_out"] + 4 for it in self.items)
        self.flops = sum(u[1] for u in self.units)
        self.launches = 4 * len(self.items)     # delayed quant, history, dgrad, wgrad
        self.config = {"workload": cfg["name"] + (f" ({only} only)" if only else ""), "M": M,
                       "linears": [[it["name"], it["n_out"], it["k_in"]] for it in self.items],
                       "scales": "per-tensor delayed (dY E5M2, X/W E4M3), history "
                                 f"{cfg['history_len']}, margin {cfg['margin']}",
                       "out": "dX bf16, dW fp32"}

    def step(self, rec=None):
        fp8, M = self.fp8, self.M
        for it in self.items:
            _run(rec, "quant:" + it["name"], lambda it=it: it["st_dy"].quantize(it["dy"], q=it["qdy"],
                                                                               update=False))
            _run(rec, "gemm:" + it["name"] + ".dgrad", lambda it=it: fp8.fp8_block_gemm(
                it["A_dg"], it["B_dg"], M, it["k_in"], it["n_out"], fp8.OUT_BF16, y=it["dx"]))
            _run(rec, "gemm:" + it["name"] + ".wgrad", lambda it=it: fp8.fp8_block_gemm(
                it["A_wg"], it["B_wg"], it["n_out"], it["k_in"], M, fp8.OUT_F32, y=it["dw"]))
            _run(rec, "quant:" + it["name"], lambda it=it: it["st_dy"].update())

    def host_io(self):
        return [it["dy"] for it in self.items], [it["dx"] for it in self.items] + [it["dw"] for it in self.items]


class MlpBwdBlock:
    """Backward of the Llama-3.1-8B MLP under the block recipe: per linear,
    dY is quantized once into its row-wise 1x128 copy (dgrad operand) and its
    column-wise transposed copy (wgrad operand) from a single read, X into
    its column-wise transposed copy; dgrad dX = dY W (W 128x128, stored
    transposed for the product, bf16 out) and wgrad dW = dY^T X (both 1x128
    along the tokens, fp32 out).  E4M3 throughout."""

    def __init__(self, cfg, fp8, device, seed=0, only=None):
        import torch
        self.fp8, self.M = fp8, cfg["M"]
        self.mode = fp8.SCALE_POW2 if cfg["scale_mode"] == "pow2" else fp8.SCALE_FP32
        M = self.M
        g = torch.Generator(device=device)
        self.items = []
        u8, f32 = torch.uint8, torch.float32
        for i, (name, n_out, k_in) in enumerate(cfg["linears"]):
            if only and name != only:
                continue
            g.manual_seed(seed * 1000 + 300 + i)
            z = _randn(g, (M, n_out), device)
            chi = sum(_randn(g, (M, n_out), device) ** 2 for _ in range(int(cfg["dy_nu"])))
            dy = (z / torch.sqrt(chi / cfg["dy_nu"]) * cfg["dy_scale"]).to(torch.bfloat16)
            del z, chi
            x = _activations(g, M, k_in, device)
            w = _randn(g, (n_out, k_in), device, 0.02).to(torch.bfloat16)
            qw, sw = fp8.fp8_quantize_128x128(w, fp8.E4M3, self.mode)   # as the forward leaves it
            it = dict(name=name, n_out=n_out, k_in=k_in, dy=dy, x=x, qw=qw, sw=sw,
                      qdy=torch.empty((M, n_out), dtype=u8, device=device),
                      sdy=torch.empty((n_out // 128, M), dtype=f32, device=device),
                      qdyt=torch.empty((n_out, M), dtype=u8, device=device),
                      sdyt=torch.empty((M // 128, n_out), dtype=f32, device=device),
                      qxt=torch.empty((k_in, M), dtype=u8, device=device),
                      sxt=torch.empty((M // 128, k_in), dtype=f32, device=device),
                      dx=torch.empty((M, k_in), dtype=torch.bfloat16, device=device),
                      dw=torch.empty((n_out, k_in), dtype=f32, device=device))
            E4 = fp8.E4M3
            it["A_dg"] = fp8.operand(it["qdy"], it["sdy"], E4, fp8.GRAN_1x128)                 # [M][n_out]
            it["B_dg"] = fp8.operand(qw, sw, E4, fp8.GRAN_128x128, transposed=True)            # W^T
            it["A_wg"] = fp8.operand(it["qdyt"], it["sdyt"], E4, fp8.GRAN_1x128)               # dY^T
            it["B_wg"] = fp8.operand(it["qxt"], it["sxt"], E4, fp8.GRAN_1x128)                 # X^T
            self.items.append(it)
        self.units = []
        for it in self.items:
            f = 2.0 * M * it["n_out"] * it["k_in"]
            qb = (4 * M * it["n_out"] + 8 * M * it["n_out"] // 128) + (3 * M * it["k_in"] + 4 * M * it["k_in"] // 128)
            self.units += [(it["name"] + ".dgrad", f, qb), (it["name"] + ".wgrad", f, 0)]
        self.flops = sum(u[1] for u in self.units)
        self.launches = 4 * len(self.items)     # dY row+col quant, X col quant, dgrad, wgrad
        self.config = {"workload": cfg["name"] + (f" ({only} only)" if only else ""), "M": M,
                       "linears": [[it["name"], it["n_out"], it["k_in"]] for it in self.items],
                       "scales": f"{cfg['scale_mode']} 1x128 (dY row-wise and column-wise, X column-wise) "
                                 "/ 128x128 (W), E4M3",
                       "out": "dX bf16, dW fp32"}

    def step(self, rec=None):
        fp8, M, mode = self.fp8, self.M, self.mode
        for it in self.items:
            n = it["name"] + ".dgrad"
            _run(rec, "quant:" + n, lambda it=it: (
                fp8.fp8_quantize_1x128_colwise(it["dy"], fp8.E4M3, mode, qt=it["qdyt"], scales_t=it["sdyt"],
                                               q=it["qdy"], scales=it["sdy"]),
                fp8.fp8_quantize_1x128_colwise(it["x"], fp8.E4M3, mode, qt=it["qxt"], scales_t=it["sxt"])))
            _run(rec, "gemm:" + n, lambda it=it: fp8.fp8_block_gemm(
                it["A_dg"], it["B_dg"], M, it["k_in"], it["n_out"], fp8.OUT_BF16, mode, y=it["dx"]))
            _run(rec, "gemm:" + it["name"] + ".wgrad", lambda it=it: fp8.fp8_block_gemm(
                it["A_wg"], it["B_wg"], it["n_out"], it["k_in"], M, fp8.OUT_F32, mode, y=it["dw"]))

    def host_io(self):
        return ([it["dy"] for it in self.items] + [it["x"] for it in self.items],
                [it["dx"] for it in self.items] + [it["dw"] for it in self.items])


class MoE:
    """Qwen3-30B-A3B-style expert GEMMs: 8192 tokens x top-8 of 128 experts
    (Zipf(1.1) loads), gate+up 2048->1536 and down 768->2048 per expert as two
    grouped block-scaled GEMMs over the expert-sorted rows."""

    def __init__(self, cfg, fp8, device, seed=0, only=None):
        import torch
        self.fp8 = fp8
        loads, off = W_.moe_routing(cfg["tokens"], cfg["experts"], cfg["topk"], cfg["zipf_a"], seed=seed)
        self.T = T = int(off[-1])
        G, H, I = cfg["experts"], cfg["hidden"], cfg["gate_up_n"]
        self.off = torch.from_numpy(off).to(device)
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000 + 500)
        self.items = []
        for name, N, K in (("gate_up", I, H), ("down", H, cfg["down_k"])):
            if only and name != only:
                continue
            x = _randn(g, (T, K), device).to(torch.bfloat16)
            w = _randn(g, (G * N, K), device, 0.02).to(torch.bfloat16)
            it = dict(name=name, N=N, K=K, x=x, w=w,
                      qx=torch.empty((T, K), dtype=torch.uint8, device=device),
                      sx=torch.empty((K // 128, T), dtype=torch.float32, device=device),
                      qw=torch.empty((G * N, K), dtype=torch.uint8, device=device),
                      sw=torch.empty((G * N // 128, K // 128), dtype=torch.float32, device=device),
                      y=torch.empty((T, N), dtype=torch.bfloat16, device=device))
            it["A"] = fp8.operand(it["qx"], it["sx"], fp8.E4M3, fp8.GRAN_1x128)
            it["B"] = fp8.operand(it["qw"], it["sw"], fp8.E4M3, fp8.GRAN_128x128)
            self.items.append(it)
        self.units = [(it["name"], 2.0 * T * it["N"] * it["K"],
                       3 * T * it["K"] + 3 * G * it["N"] * it["K"]) for it in self.items]
        self.flops = sum(u[1] for u in self.units)
        self.launches = 3 * len(self.items)
        self.config = {"workload": cfg["name"] + (f" ({only} only)" if only else ""), "rows": T,
                       "experts": G, "max_rows": int(loads.max()), "min_rows": int(loads.min()),
                       "linears": [[it["name"], it["N"], it["K"]] for it in self.items],
                       "scales": "fp32 1x128 (X) / 128x128 (W)", "out": "bf16"}

    def step(self, rec=None):
        fp8, T = self.fp8, self.T
        for it in self.items:
            # the stacked [G*N][K] weights quantize per expert tile since N % 128 == 0
            _run(rec, "quant:" + it["name"], lambda it=it: fp8.fp8_quantize_linear(
                it["x"], it["w"], qx=it["qx"], sx=it["sx"], qw=it["qw"], sw=it["sw"]))
            _run(rec, "gemm:" + it["name"], lambda it=it: fp8.fp8_grouped_block_gemm(
                self.off, it["A"], it["B"], T, it["N"], it["K"], fp8.OUT_BF16, y=it["y"]))

    def host_io(self):
        return [it["x"] for it in self.items] + [it["w"] for it in self.items], [it["y"] for it in self.items]


class FusedMlp:
    """An MLP block as two chained FP8 linears whose intermediate stays FP8:
    quant X (1x128) and re-quant W_gate_up, W_down (128x128); the gate/up
    product's epilogue applies SwiGLU and quantizes to the down product's
    1x128 operand (no bf16 intermediate, no separate quantization pass);
    the down product writes bf16.  Dense (Llama-3.1-8B MLP) or grouped
    (Qwen3-30B-A3B experts, Zipf(1.1) loads)."""

    def __init__(self, cfg, fp8, device, seed=0, only=None):
        import torch
        self.fp8 = fp8
        self.mode = fp8.SCALE_POW2 if cfg["scale_mode"] == "pow2" else fp8.SCALE_FP32
        D, I = cfg["hidden"], cfg["intermediate"]
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000 + 700)
        if "experts" in cfg:
            loads, off = W_.moe_routing(cfg["tokens"], cfg["experts"], cfg["topk"], cfg["zipf_a"],
                                        seed=seed)
            self.off = torch.from_numpy(off).to(device)
            rows, G = int(off[-1]), cfg["experts"]
            self.x = _randn(g, (rows, D), device).to(torch.bfloat16)
            extra = {"rows": rows, "experts": G, "max_rows": int(loads.max()), "min_rows": int(loads.min())}
        else:
            self.off = None
            rows, G = cfg["M"], 1
            self.x = _activations(g, rows, D, device)
            extra = {"M": rows}
        self.rows, self.D, self.I, self.G = rows, D, I, G
        # per expert: W_gate_up [2I][D] (I gate rows, then I up rows), W_down [D][I]
        self.w_gu = _randn(g, (G * 2 * I, D), device, 0.02).to(torch.bfloat16)
        self.w_dn = _randn(g, (G * D, I), device, 0.02).to(torch.bfloat16)
        u8, f32 = torch.uint8, torch.float32
        self.qx = torch.empty((rows, D), dtype=u8, device=device)
        self.sx = torch.empty((D // 128, rows), dtype=f32, device=device)
        self.qgu = torch.empty((G * 2 * I, D), dtype=u8, device=device)
        self.sgu = torch.empty((G * 2 * I // 128, D // 128), dtype=f32, device=device)
        self.qdn = torch.empty((G * D, I), dtype=u8, device=device)
        self.sdn = torch.empty((G * D // 128, I // 128), dtype=f32, device=device)
        self.qh = torch.empty((rows, I), dtype=u8, device=device)
        self.sh = torch.empty((I // 128, rows), dtype=f32, device=device)
        self.y = torch.empty((rows, D), dtype=torch.bfloat16, device=device)
        E4 = fp8.E4M3
        self.A_gu = fp8.operand(self.qx, self.sx, E4, fp8.GRAN_1x128)
        self.B_gu = fp8.operand(self.qgu, self.sgu, E4, fp8.GRAN_128x128)
        self.A_dn = fp8.operand(self.qh, self.sh, E4, fp8.GRAN_1x128)
        self.B_dn = fp8.operand(self.qdn, self.sdn, E4, fp8.GRAN_128x128)
        self.units = [("gate_up", 2.0 * rows * 2 * I * D,
                       3 * rows * D + 4 * rows * (D // 128) + 3 * G * 2 * I * D + 4 * G * 2 * I * D // 16384),
                      ("down", 2.0 * rows * D * I, 3 * G * D * I + 4 * G * D * I // 16384)]
        self.flops = sum(u[1] for u in self.units)
        self.launches = 5
        self.config = {"workload": cfg["name"], **extra, "hidden": D, "intermediate": I,
                       "linears": [["gate_up+swiglu", 2 * I, D], ["down", D, I]],
                       "scales": f"{cfg['scale_mode']} 1x128 (X, h) / 128x128 (W)",
                       "out": "h: e4m3 + 1x128 scales from the gate/up epilogue; y: bf16"}

    def step(self, rec=None):
        fp8, mode, rows, D, I = self.fp8, self.mode, self.rows, self.D, self.I
        _run(rec, "quant:gate_up", lambda: (
            fp8.fp8_quantize_1x128(self.x, fp8.E4M3, mode, q=self.qx, scales=self.sx),
            fp8.fp8_quantize_128x128(self.w_gu, fp8.E4M3, mode, q=self.qgu, scales=self.sgu)))
        if self.off is None:
            _run(rec, "gemm:gate_up", lambda: fp8.fp8_block_gemm_quant(
                self.A_gu, self.B_gu, rows, 2 * I, D, fp8.EPI_SWIGLU, fp8.E4M3, mode, mode,
                q=self.qh, q_scales=self.sh))
        else:
            _run(rec, "gemm:gate_up", lambda: fp8.fp8_grouped_block_gemm_quant(
                self.off, self.A_gu, self.B_gu, rows, 2 * I, D, fp8.EPI_SWIGLU, fp8.E4M3, mode, mode,
                q=self.qh, q_scales=self.sh))
        _run(rec, "quant:down", lambda: fp8.fp8_quantize_128x128(self.w_dn, fp8.E4M3, mode, q=self.qdn,
                                                                 scales=self.sdn))
        if self.off is None:
            _run(rec, "gemm:down", lambda: fp8.fp8_block_gemm(
                self.A_dn, self.B_dn, rows, D, I, fp8.OUT_BF16, mode, y=self.y))
        else:
            _run(rec, "gemm:down", lambda: fp8.fp8_grouped_block_gemm(
                self.off, self.A_dn, self.B_dn, rows, D, I, fp8.OUT_BF16, mode, y=self.y))

    def host_io(self):
        return [self.x, self.w_gu, self.w_dn], [self.y]


class Attn:
    """Llama-3.1-8B attention prefill over an FP8 KV cache: quantize Q (1x128:
    one scale per token and head), write the KV cache (K and V quantized
    128x128: one scale per 128 tokens and head), FP8 attention forward
    (causal, GQA 32/8 heads, head_dim 128) -> O bf16."""

    def __init__(self, cfg, fp8, device, seed=0, only=None):
        import torch
        self.fp8 = fp8
        S, hq, hkv = cfg["seq"], cfg["heads_q"], cfg["heads_kv"]
        self.S, self.hq, self.hkv = S, hq, hkv
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000 + 900)
        self.q = _randn(g, (S, hq * 128), device).to(torch.bfloat16)
        self.k = _randn(g, (S, hkv * 128), device).to(torch.bfloat16)
        self.v = _randn(g, (S, hkv * 128), device).to(torch.bfloat16)
        u8, f32 = torch.uint8, torch.float32
        self.qq = torch.empty((S, hq * 128), dtype=u8, device=device)
        self.sq = torch.empty((hq, S), dtype=f32, device=device)
        self.kq = torch.empty((S, hkv * 128), dtype=u8, device=device)
        self.sk = torch.empty(((S + 127) // 128, hkv), dtype=f32, device=device)
        self.vq = torch.empty((S, hkv * 128), dtype=u8, device=device)
        self.sv = torch.empty(((S + 127) // 128, hkv), dtype=f32, device=device)
        self.o = torch.empty((S, hq * 128), dtype=torch.bfloat16, device=device)
        self.Q = fp8.attn_input(self.qq, self.sq)
        self.K = fp8.attn_input(self.kq, self.sk)
        self.V = fp8.attn_input(self.vq, self.sv)
        pairs = S * (S + 1) // 2 if cfg["causal"] else S * S
        self.causal = cfg["causal"]
        qbytes = 3 * S * (hq + 2 * hkv) * 128 + 4 * S * hq + 8 * ((S + 127) // 128) * hkv
        self.units = [("attn", 4.0 * 128 * hq * pairs, qbytes)]
        self.flops = self.units[0][1]
        self.launches = 4
        self.config = {"workload": cfg["name"], "seq": S, "heads_q": hq, "heads_kv": hkv, "head_dim": 128,
                       "causal": bool(cfg["causal"]),
                       "scales": "Q 1x128 (token, head); K, V 128x128 (128 tokens, head); P E4M3 / 448",
                       "out": "bf16", "flops": "4 * 128 * heads_q * visible (query, key) pairs"}

    def step(self, rec=None):
        fp8 = self.fp8
        _run(rec, "quant:attn", lambda: (
            fp8.fp8_quantize_1x128(self.q, q=self.qq, scales=self.sq),
            fp8.fp8_quantize_128x128(self.k, q=self.kq, scales=self.sk),
            fp8.fp8_quantize_128x128(self.v, q=self.vq, scales=self.sv)))
        _run(rec, "gemm:attn", lambda: fp8.fp8_attention_fwd(
            self.Q, self.K, self.V, self.S, self.S, self.hq, self.hkv, self.causal, 128 ** -0.5, o=self.o))

    def host_io(self):
        return [self.q, self.k, self.v], [self.o]


WORKLOADS = {"llama3.1-8b-fprop": (Fprop, W_.LLAMA31_8B_FPROP),
             "llama3.1-8b-fprop-mxfp8": (Fprop, W_.LLAMA31_8B_FPROP_MX),
             "llama2-7b-fprop": (Fprop, W_.LLAMA2_7B_FPROP),
             "tiny-fprop": (Fprop, W_.TINY_FPROP),
             "llama3.1-8b-mlp-bwd": (MlpBwd, W_.LLAMA31_8B_MLP_BWD),
             "llama3.1-8b-mlp-bwd-blockwise": (MlpBwdBlock, W_.LLAMA31_8B_MLP_BWD_BLOCK),
             "qwen3-30b-a3b-moe": (MoE, W_.QWEN3_30B_MOE),
             "llama3.1-8b-mlp-fused": (FusedMlp, W_.LLAMA31_8B_MLP_FUSED),
             "qwen3-30b-a3b-moe-fused": (FusedMlp, W_.QWEN3_30B_MOE_FUSED),
             "llama3.1-8b-attn-fp8": (Attn, W_.LLAMA31_8B_ATTN)}


# ------------------------------------------------------------ CPU oracle
def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _par(fn, jobs, n):
    """fn(job) for every job on n host threads.  The oracle's C routines are
    called through ctypes, which releases the GIL, so the threads run on
    separate cores."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=n) as ex:
        return list(ex.map(fn, jobs))


def _chunks(n, parts, align=1):
    step = max(align, -(-n // parts) // align * align)
    return [(i, min(n, i + step)) for i in range(0, n, step)]


def oracle_linear(orc, x, w, mode, mx, threads, gemm_rows, w_rows=None):
    """The oracle on one FP8 linear: quantize X (1x128, or 1x32 for MXFP8) and
    W (128x128, or 1x32) -- rows split over `threads` host threads -- then the
    fp64 product of the first `gemm_rows` rows of X with the quantized rows of
    W (all of W, or its first `w_rows`).  x, w: bf16 bit patterns.  Returns
    (quantization seconds, product seconds, product flops)."""
    K = x.shape[1]
    if w_rows is not None:
        w = w[:w_rows]
    N = w.shape[0]
    qx_fn = (lambda a: orc.quantize_mx(a)) if mx else (lambda a: orc.quantize_1x128(a, orc.E4M3, mode))
    qw_fn = (lambda a: orc.quantize_mx(a)) if mx else (lambda a: orc.quantize_128x128(a, orc.E4M3, mode))
    xc = _chunks(x.shape[0], threads)
    wc = _chunks(N, threads, 128)
    t0 = time.perf_counter()
    rx = _par(lambda c: qx_fn(x[c[0]:c[1]]), xc, threads)
    rw = _par(lambda c: qw_fn(w[c[0]:c[1]]), wc, threads)
    t1 = time.perf_counter()
    qw = np.concatenate([q for q, _ in rw], axis=0)
    sw = np.concatenate([s for _, s in rw], axis=0) if not mx else np.concatenate([s for _, s in rw], axis=1)
    qx = np.concatenate([q for q, _ in rx], axis=0)[:gemm_rows]
    sx = np.concatenate([s for _, s in rx], axis=1)[:, :gemm_rows]
    gx = orc.GRAN_1x32 if mx else orc.GRAN_1x128
    gw = orc.GRAN_1x32 if mx else orc.GRAN_128x128
    A = orc.operand(qx, orc.E4M3, gx, np.ascontiguousarray(sx))
    B = orc.operand(qw, orc.E4M3, gw, np.ascontiguousarray(sw))
    t2 = time.perf_counter()
    _par(lambda c: orc.gemm(gemm_rows, N, K, A, B, rows=np.arange(c[0], c[1])),
         _chunks(gemm_rows, threads), threads)
    t3 = time.perf_counter()
    return t1 - t0, t3 - t2, 2.0 * gemm_rows * N * K


def cpu_oracle_baseline(wl, gemm_rows=256):
    """The oracle on the host cores for one step of an fprop workload: every X
    and W quantized in full (timed), the product on the first `gemm_rows`
    rows of each X with all columns (timed), the product's time extrapolated
    linearly to all rows.  Returns the cpu_baseline object (step TFLOP/s)."""
    import oracle as orc
    n = host_threads()
    mode = orc.SCALE_POW2 if wl.mode == wl.fp8.SCALE_POW2 else orc.SCALE_FP32
    tq = tg = tg_full = 0.0
    for it in wl.items:
        import torch
        x = it["x"].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        w = it["w"].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        q_s, g_s, _ = oracle_linear(orc, x, w, mode, wl.mx, n, gemm_rows)
        tq += q_s
        tg += g_s
        tg_full += g_s * wl.M / gemm_rows
    secs = tq + tg_full
    return {"value": wl.flops / secs / 1e12, "unit": "TFLOP/s", "cores": n, "kind": "oracle",
            "seconds_measured": tq + tg, "seconds_step_extrapolated": secs,
            "quant_seconds": tq, "gemm_seconds_sample": tg,
            "sample": f"per linear: X and W quantized in full (measured); product on {gemm_rows} rows x all "
                      f"columns in fp64 (measured), its time x {wl.M // gemm_rows} for all rows "
                      f"(extrapolated); {n} host threads"}


# ------------------------------------------------------------------ arms
REF_X_ROWS, REF_W_ROWS = 64, 512


def run_reference(args):
    """The oracle as it stands on this host's cores, on the fprop workload's
    config; each step is a bounded sample of it: per linear, 64 X rows
    quantized (1x128, or 1x32 for MXFP8), 512 W rows quantized (128x128, or
    1x32) and the 64 x 512 block of Y in fp64, work split over every host
    thread."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle as orc
    cls, cfg = WORKLOADS[args.workload]
    if cls is not Fprop:
        print(json.dumps({"impl": "reference", "unavailable":
                          "the reference arm samples the fprop workloads only"}), flush=True)
        return 0
    mode = orc.SCALE_POW2 if cfg["scale_mode"] in ("pow2", "mx") else orc.SCALE_FP32
    mx = cfg["scale_mode"] == "mx"
    n = host_threads()
    lin = [(W_.activations(REF_X_ROWS, K, seed=1), W_.gaussian((min(REF_W_ROWS, N), K), 0.02, seed=2))
           for name, N, K in cfg["linears"] if not args.only or name == args.only]

    def step():
        f = 0.0
        for x, w in lin:
            f += oracle_linear(orc, x, w, mode, mx, n, REF_X_ROWS)[2]
        return f

    for _ in range(args.warmup):
        step()
    times, fl = [], 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        fl = step()
        times.append(time.perf_counter() - t0)
    dt = float(np.median(times))
    val = fl / dt / 1e12
    sample = (f"per linear: {REF_X_ROWS} X rows and {REF_W_ROWS} W rows quantized "
              f"({'1x32' if mx else '1x128 / 128x128'}), the {REF_X_ROWS}x{REF_W_ROWS} block of Y in fp64; "
              f"{n} host threads; median step")
    config = dict(Fprop.static_config(cfg, args.only))
    config.update(bench_config_extra(ws))
    line = {"metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": config,
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": n, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def bench_config_extra(ws):
    return {"l2": f"flushed between steps ({FLUSH_BYTES >> 20} MiB write); every step also streams "
                  "> 129 MB of inputs", "timing": "median of per-step CUDA-event times",
            "parallelism": f"replicas x{ws}"}


def run_ours(args):
    import torch
    import block_scaled_gemm_quantize_gb300 as fp8
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    fp8.lib()
    peaks = _peaks()
    cls, cfg = WORKLOADS[args.workload]
    wl = cls(cfg, fp8, device, seed=rank, only=args.only)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(v):
        return reduce_max(v, device)

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def l2_flush():   # a write larger than L2 between steps (outside the step's events)
        flush.fill_(1)

    for _ in range(args.warmup):
        l2_flush()
        wl.step()
    torch.cuda.synchronize()

    # --- timed region: K steps, an L2 flush before each, per-step and
    # per-phase events on the launching stream; the step time is the median
    rec = Rec()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    step_ev = []
    t_start.record()
    for s in range(args.steps):
        l2_flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        rec.step = s
        e0.record()
        wl.step(rec)
        e1.record()
        step_ev.append((e0, e1))
    t_end.record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    fp8.device_status()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in step_ev]
    ms = max_over_ranks(float(np.median(step_ms)))
    wall_ms = max_over_ranks(t_start.elapsed_time(t_end)) / args.steps
    tot = rec.medians()

    per = []
    gemm_ms = 0.0
    gemm_flops = 0.0
    for name, fl, qb in wl.units:
        g = tot.get("gemm:" + name, 0.0)
        q = tot.get("quant:" + name, 0.0)
        gemm_ms += g
        gemm_flops += fl
        e = {"unit": name, "gemm_us": g * 1e3, "gemm_tflops": fl / g / 1e9 if g else None}
        if q:
            e.update({"quant_us": q * 1e3, "quant_gbs": qb / q / 1e6 if qb else None})
        per.append(e)
    quant_ms = sum(v for k, v in tot.items() if k.startswith("quant:"))
    qbytes = getattr(wl, "quant_bytes", None) or sum(u[2] for u in wl.units)
    achieved = gemm_flops / gemm_ms / 1e9
    digest = kernel_digest()
    tr = GEMM_TRAFFIC["bytes"].get(args.workload) if GEMM_TRAFFIC["sources_sha256"] == digest else None
    traffic = (sum(tr[u[0]] for u in wl.units) / len(wl.units)
               if tr and all(u[0] in tr for u in wl.units) else None)
    # the products are timed in launches of 0.1-1 ms at the maximum SM clock: the burst peak
    fp8_peak = FP8_OVER_BF16 * peaks["bf16"]
    fp8_peak_sustained = FP8_OVER_BF16 * peaks["bf16_sustained"]
    quant_gbs = qbytes / quant_ms / 1e6 if quant_ms else None

    # --- end to end through host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        # End to end through pinned host buffers: every step copies its inputs
        # host -> device and its outputs device -> host.  Copies run on their
        # own streams so that, unit by unit (a linear of the fprop step; the
        # whole step otherwise), the next unit's inputs upload and the previous
        # unit's outputs download while this unit computes.  Per-unit events
        # keep a buffer from being overwritten before the step that reads it
        # (or the copy that reads it back) is done.
        units = wl.e2e_units() if hasattr(wl, "e2e_units") else \
            [(wl.host_io()[0], wl.host_io()[1], wl.step)]
        h_units = [([t.cpu().pin_memory() for t in ins], [torch.empty(t.shape, dtype=t.dtype).pin_memory()
                                                            for t in outs]) for ins, outs, _ in units]
        h2d = sum(t.numel() * t.element_size() for hi, _ in h_units for t in hi)
        d2h = sum(t.numel() * t.element_size() for _, ho in h_units for t in ho)
        s_h2d, s_cmp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev_c = [torch.cuda.Event() for _ in units]
        ev_d = [torch.cuda.Event() for _ in units]
        for e in ev_c + ev_d:
            e.record()

        def e2e_step():
            ev_h = []
            for i, (ins, _, _) in enumerate(units):
                s_h2d.wait_event(ev_c[i])               # the previous step has read these inputs
                with torch.cuda.stream(s_h2d):
                    for h, d in zip(h_units[i][0], ins):
                        d.copy_(h, non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_h2d)
                ev_h.append(e)
            for i, (_, outs, fn) in enumerate(units):
                s_cmp.wait_event(ev_h[i])
                s_cmp.wait_event(ev_d[i])               # the previous step's outputs are read back
                with torch.cuda.stream(s_cmp):
                    fn()
                ev_c[i].record(s_cmp)
                s_d2h.wait_event(ev_c[i])
                with torch.cuda.stream(s_d2h):
                    for h, d in zip(h_units[i][1], outs):
                        h.copy_(d, non_blocking=True)
                ev_d[i].record(s_d2h)

        e2e_steps = max(3, min(args.steps, 20))
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        main = torch.cuda.current_stream()
        a.record(main)
        for st in (s_h2d, s_cmp, s_d2h):
            st.wait_stream(main)
        for _ in range(e2e_steps):
            e2e_step()
        for st in (s_h2d, s_cmp, s_d2h):
            main.wait_stream(st)
        b.record(main)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b)) / e2e_steps
        e2e = {"value": wl.flops * ws / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": e2e_steps, "overlap": f"{len(units)} unit(s) per step, copy and compute streams"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and cls is Fprop:
        cpu = cpu_oracle_baseline(wl)

    value = wl.flops * ws / (ms * 1e-3) / 1e12
    config = dict(wl.config)
    config.update(bench_config_extra(ws))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_wall": wall_ms,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3/e5m2 (fp32 accumulate)", "data": "synthetic",
        "config": config,
        "pct_of_fp8_peak": 100.0 * value / fp8_peak,
        "roofline": {"bound": "tensor", "kernel": dominant_kernel(wl), "achieved": achieved,
                     "peak": fp8_peak, "unit": "TFLOP/s", "frac": achieved / fp8_peak,
                     "traffic": traffic, "traffic_unit": "DRAM bytes per launch (mean, ncu)",
                     "kernel_sources_sha256": digest,
                     "peak_src": f"{peaks['src']}: 2 x bf16_tflops, burst ({peaks['bf16']})",
                     "frac_of_sustained_peak": achieved / fp8_peak_sustained},
        "quant_roofline": {"bound": "hbm", "achieved": quant_gbs, "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": quant_gbs / peaks["hbm_gbs"] if quant_gbs else None},
        "per_unit": per,
        "clocks": clk,
        "gpu_launches": wl.launches * args.steps,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="llama3.1-8b-fprop")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None, help="run a single linear of the workload (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
