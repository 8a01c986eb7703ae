"""Multi-process paths on CPU with the gloo backend (world size 2):
- the data-parallel exchange of delayed scaling (MAX of the per-rank amax),
  checked against the single-process oracle trajectory of the whole tensor;
- the benchmark's max-over-ranks timing reduction."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, fn, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, fn(rank, world)))
    finally:
        dist.destroy_process_group()


def _run(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, fn, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


STEPS, ROWS, COLS = 6, 64, 256


def _dp_delayed(rank, world):
    import block_scaled_gemm_quantize_gb300 as fp8
    st = orc.DelayedState(4, orc.E5M2, margin=0)
    scales = []
    for t in range(STEPS):
        x = inputs.student_t((ROWS, COLS), 3.0, 1e-3 * (1 + t % 3), seed=300 + t)
        shard = x[rank * ROWS // world:(rank + 1) * ROWS // world]
        _, amax = orc.quantize_tensor(np.ascontiguousarray(shard), orc.E5M2, float(st.scale[0]))
        a = torch.tensor([amax], dtype=torch.float32)
        fp8.reduce_amax(a)                       # the binding's exchange step
        st.update(float(a[0]))
        scales.append(float(st.scale[0]))
    return scales


def test_data_parallel_amax_exchange_matches_single_process():
    out = _run(_dp_delayed)
    ref = orc.DelayedState(4, orc.E5M2, margin=0)
    want = []
    for t in range(STEPS):
        x = inputs.student_t((ROWS, COLS), 3.0, 1e-3 * (1 + t % 3), seed=300 + t)
        ref.step(x)
        want.append(float(ref.scale[0]))
    assert out[0] == out[1] == want


def _bench_reduce(rank, world):
    import bench
    return bench.reduce_max(10.0 + rank * 5.0, "cpu")


def test_bench_max_over_ranks():
    out = _run(_bench_reduce)
    assert out == {0: 15.0, 1: 15.0}
