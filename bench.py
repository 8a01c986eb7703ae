#!/usr/bin/env python
"""Benchmark of the FP8 linear layer on GB300: block quantization + block-scaled
FP8 GEMM, reported as quant+GEMM TFLOP/s of the Llama-3.1-8B-shaped fprop
linears (M = 8192 tokens; QKV 4096->6144, O 4096->4096, gate+up 4096->28672,
down 14336->4096; X per 1x128, W per 128x128, E4M3, fp32 scales, bf16 out).

One step = for each linear: quantize X (1x128), re-quantize W (128x128, the
weights change every optimizer step), GEMM -> Y bf16.  Inputs are synthetic
(seeded, X ~ N(0,1) with 1% outlier channels x20, W ~ N(0, 0.02)), resident
in HBM; the step streams ~1.2 GB, larger than the 129 MB L2.

  python bench.py [--steps K] [--warmup W] [--impl ours|reference]
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_scaled_gemm_quantize_gb300 import inputs as W_  # noqa: E402

WORKLOAD = W_.LLAMA31_8B_FPROP
METRIC = "block-scaled FP8 linear TFLOPS (quant+GEMM) and % of GB300 dense FP8 peak"
FP8_OVER_BF16 = 2.0      # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


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


# ------------------------------------------------------------ workload
def make_inputs(device, seed=0, only=None):
    """Synthetic bf16 inputs on the device, per linear: X [M, K], W [N, K]."""
    import torch
    g = torch.Generator(device=device)
    M = WORKLOAD["M"]
    bufs = []
    for i, (name, N, K) in enumerate(WORKLOAD["linears"]):
        if only and name != only:
            continue
        g.manual_seed(seed * 1000 + i)
        x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
        n_out = int(round(0.01 * K))
        cols = torch.randperm(K, generator=g, device=device)[:n_out]
        x[:, cols] *= 20.0
        w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * 0.02
        bufs.append((name, N, K, x.to(torch.bfloat16), w.to(torch.bfloat16)))
        del x, w
    return bufs


class Step:
    """Preallocated quant+GEMM pass over every linear of the workload."""

    def __init__(self, bufs, fp8, device):
        import torch
        self.fp8, self.items = fp8, []
        M = WORKLOAD["M"]
        for name, N, K, x, w in bufs:
            qx = torch.empty((M, K), dtype=torch.uint8, device=device)
            sx = torch.empty((K // 128, M), dtype=torch.float32, device=device)
            qw = torch.empty((N, K), dtype=torch.uint8, device=device)
            sw = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=device)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
            A = fp8.operand(qx, sx, fp8.E4M3, fp8.GRAN_1x128)
            B = fp8.operand(qw, sw, fp8.E4M3, fp8.GRAN_128x128)
            self.items.append(dict(name=name, N=N, K=K, x=x, w=w, qx=qx, sx=sx, qw=qw, sw=sw, y=y,
                                   A=A, B=B))
        self.M = M
        self.flops = sum(2.0 * M * it["N"] * it["K"] for it in self.items)
        self.launches = 3 * len(self.items)

    def run(self, ev=None):
        fp8, M = self.fp8, self.M
        for i, it in enumerate(self.items):
            if ev is not None:
                ev[i][0].record()
            fp8.fp8_quantize_1x128(it["x"], fp8.E4M3, fp8.SCALE_FP32, q=it["qx"], scales=it["sx"])
            fp8.fp8_quantize_128x128(it["w"], fp8.E4M3, fp8.SCALE_FP32, q=it["qw"], scales=it["sw"])
            if ev is not None:
                ev[i][1].record()
            fp8.fp8_block_gemm(it["A"], it["B"], M, it["N"], it["K"], fp8.OUT_BF16, fp8.SCALE_FP32,
                               y=it["y"])
            if ev is not None:
                ev[i][2].record()


def quant_bytes(M, N, K):
    """Algorithmic bytes of the two quantizers of one linear: bf16 read,
    one code byte written, one fp32 scale per 1x128 / 128x128 tile."""
    x = M * K * 3 + 4 * M * (K // 128)
    w = N * K * 3 + 4 * ((N + 127) // 128) * (K // 128)
    return x + w


# ------------------------------------------------------------ CPU oracle
def cpu_oracle_sample(rows_x, w_bits, xs_bits, rows=8):
    """Time the oracle on a bounded sample: per linear, quantize the full W
    (128x128) and `rows` rows of X (1x128), and compute those rows of Y in
    fp64.  Returns (seconds, flops of the sample)."""
    import oracle as orc
    t0 = time.perf_counter()
    flops = 0.0
    for x, w in zip(xs_bits, w_bits):
        N, K = w.shape
        qw, sw = orc.quantize_128x128(w)
        qx, sx = orc.quantize_1x128(x[:rows])
        A = orc.operand(qx, orc.E4M3, orc.GRAN_1x128, sx)
        B = orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw)
        orc.gemm(rows, N, K, A, B)
        flops += 2.0 * rows * N * K
    return time.perf_counter() - t0, flops


def host_sample(bufs, rows):
    import torch
    xs, ws = [], []
    for _, N, K, x, w in bufs:
        xs.append(x[:rows].contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
        ws.append(w.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
    return xs, ws


# ------------------------------------------------------------------ arms
def run_reference(args):
    """The oracle as it stands on this host's cores; each step is a bounded
    sample of the workload (per linear: 128 rows of W quantized 128x128, 4 rows
    of X quantized 1x128, those 4 rows x 128 columns of Y in fp64)."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle as orc
    rng = np.random.default_rng(0)
    lin = []
    for name, N, K in WORKLOAD["linears"]:
        x = W_.activations(4, K, seed=1)
        w = W_.gaussian((128, K), 0.02, seed=2)
        lin.append((x, w, K))

    def step():
        f = 0.0
        for x, w, K in lin:
            qw, sw = orc.quantize_128x128(w)
            qx, sx = orc.quantize_1x128(x)
            orc.gemm(4, 128, K, orc.operand(qx, orc.E4M3, orc.GRAN_1x128, sx),
                     orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw))
            f += 2.0 * 4 * 128 * K
        return f

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += step()
    dt = time.perf_counter() - t0
    val = fl / dt / 1e12
    sample = "per linear: 128 W rows (128x128), 4 X rows (1x128), 4x128 outputs in fp64"
    line = {"metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": WORKLOAD["name"], "M": WORKLOAD["M"],
                       "linears": WORKLOAD["linears"], "sample": sample},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


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

    bufs = make_inputs(device, seed=rank, only=args.only)
    step = Step(bufs, fp8, device)
    nlin = len(step.items)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(v):
        if ws == 1:
            return v
        import torch.distributed as dist
        t = torch.tensor([v], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()

    # --- timed region: K steps, per-kernel events on the launching stream
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nlin)]
           for _ in range(args.steps)]
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for k in range(args.steps):
        step.run(evs[k])
    t_end.record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    fp8.device_status()
    ms = max_over_ranks(t_start.elapsed_time(t_end)) / args.steps

    gemm_ms = np.zeros(nlin)
    quant_ms = np.zeros(nlin)
    for k in range(args.steps):
        for i in range(nlin):
            quant_ms[i] += evs[k][i][0].elapsed_time(evs[k][i][1])
            gemm_ms[i] += evs[k][i][1].elapsed_time(evs[k][i][2])
    gemm_ms /= args.steps
    quant_ms /= args.steps
    M = WORKLOAD["M"]
    per_linear = []
    for i, it in enumerate(step.items):
        fl = 2.0 * M * it["N"] * it["K"]
        qb = quant_bytes(M, it["N"], it["K"])
        per_linear.append({"linear": it["name"], "M": M, "N": it["N"], "K": it["K"],
                           "gemm_us": gemm_ms[i] * 1e3, "gemm_tflops": fl / gemm_ms[i] / 1e9,
                           "quant_us": quant_ms[i] * 1e3, "quant_gbs": qb / quant_ms[i] / 1e6})
    gemm_flops = sum(2.0 * M * it["N"] * it["K"] for it in step.items)
    achieved = gemm_flops / gemm_ms.sum() / 1e9                     # TFLOP/s
    fp8_peak = FP8_OVER_BF16 * peaks["bf16_sustained"]
    qbytes = sum(quant_bytes(M, it["N"], it["K"]) for it in step.items)
    quant_gbs = qbytes / quant_ms.sum() / 1e6

    # --- end to end through host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        hx = [it["x"].cpu().pin_memory() for it in step.items]
        hw = [it["w"].cpu().pin_memory() for it in step.items]
        hy = [torch.empty(it["y"].shape, dtype=it["y"].dtype).pin_memory() for it in step.items]
        h2d = sum(t.numel() * 2 for t in hx + hw)
        d2h = sum(t.numel() * 2 for t in hy)

        def e2e_step():
            for i, it in enumerate(step.items):
                it["x"].copy_(hx[i], non_blocking=True)
                it["w"].copy_(hw[i], non_blocking=True)
            step.run()
            for i, it in enumerate(step.items):
                hy[i].copy_(it["y"], non_blocking=True)

        e2e_steps = max(3, min(args.steps, 20))
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(e2e_steps):
            e2e_step()
        b.record()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b)) / e2e_steps
        e2e = {"value": step.flops * ws / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": e2e_steps}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        xs, wsb = host_sample(bufs, rows=8)
        secs, fl = cpu_oracle_sample(None, wsb, xs, rows=8)
        cpu = {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "seconds": secs,
               "sample": "per linear: full W quantized 128x128, 8 X rows quantized 1x128, "
                         "8 full rows of Y in fp64 (single-threaded C oracle)"}

    value = step.flops * ws / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
        "config": {"workload": WORKLOAD["name"] + (f" ({args.only} only)" if args.only else ""),
                   "M": M, "linears": [list(l) for l in WORKLOAD["linears"]
                                       if not args.only or l[0] == args.only],
                   "scales": "fp32 1x128 (X) / 128x128 (W)", "out": "bf16",
                   "l2": "inputs larger than L2 (each step streams ~1.2 GB)",
                   "parallelism": f"replicas x{ws}"},
        "pct_of_fp8_peak": 100.0 * value / fp8_peak,
        "roofline": {"bound": "tensor", "kernel": "k_fp8_gemm", "achieved": achieved,
                     "peak": fp8_peak, "unit": "TFLOP/s", "frac": achieved / fp8_peak,
                     "traffic": None,
                     "peak_src": f"{peaks['src']}: 2 x bf16_tflops_sustained "
                                 f"({peaks['bf16_sustained']})"},
        "quant_roofline": {"bound": "hbm", "achieved": quant_gbs, "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": quant_gbs / peaks["hbm_gbs"]},
        "per_linear": per_linear,
        "clocks": clk,
        "gpu_launches": step.launches * args.steps,
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
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=[l[0] for l in WORKLOAD["linears"]], default=None,
                    help="run a single linear of the workload (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
