"""The Qwen3-30B-A3B-style mixture-of-experts expert products at full size, as
the benchmark runs them ("NVIDIA NeMo RL logra una aceleracion del 48%...",
hotbookzone.com, "Ganancias de rendimiento en el mundo real": the FP8 recipe
on a Qwen3-30B mixture-of-experts model): 8192 tokens routed top-8 over 128
experts with seeded Zipf(1.1) loads (65536 expert-sorted rows, groups of 88
to 7340 rows), X per 1x128 and the experts' weights per 128x128 tile (E4M3,
fp32 scales), one grouped product for gate+up (2048 -> 1536) and one for down
(768 -> 2048), bf16 out.

Checked against the oracle on 256 sampled rows of each of the 8 largest
experts plus every row of 8 randomly chosen small experts (fewer than 128
rows), on one sampled column per 128-column block; the fused form (SwiGLU and
quantization to the down product's operand in the gate+up epilogue) on 32
rows of the 8 largest experts and every row of 2 small ones, all columns."""
import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import (dev, host, par_grouped_gemm, par_quantize_1x128, par_quantize_128x128,
                     stratified)

pytestmark = pytest.mark.gpu
REL = 1e-5
TOKENS, EXPERTS, TOPK, ZIPF = 8192, 128, 8, 1.1
HIDDEN, INTER = 2048, 768


@pytest.fixture(scope="module")
def routing():
    loads, off = inputs.moe_routing(TOKENS, EXPERTS, TOPK, ZIPF, seed=0)
    assert int(off[-1]) == TOKENS * TOPK and loads.min() > 0
    return loads, off


def _sample_rows(loads, off, rng, big_rows, n_small):
    order = np.argsort(-loads, kind="stable")
    rows = []
    for g in order[:8]:
        rows.append(off[g] + np.sort(rng.choice(loads[g], size=min(big_rows, loads[g]), replace=False)))
    small = np.flatnonzero(loads < 128)
    for g in rng.choice(small, size=min(n_small, small.size), replace=False):
        rows.append(np.arange(off[g], off[g + 1]))
    return np.unique(np.concatenate(rows)).astype(np.int64)


def _operands(T, N, K, seed):
    x = inputs.gaussian((T, K), 1.0, seed=seed)
    w = inputs.gaussian((EXPERTS * N, K), 0.02, seed=seed + 1)
    qa, sa = par_quantize_1x128(orc, x, orc.E4M3, orc.SCALE_FP32)
    qw, sw = par_quantize_128x128(orc, w, orc.E4M3, orc.SCALE_FP32)
    sw = sw.reshape(EXPERTS, N // 128, K // 128)
    A_o = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B_o = orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw)
    A_d = fp8.operand(dev(qa), dev(sa))
    B_d = fp8.operand(dev(qw), dev(sw), gran=fp8.GRAN_128x128)
    return A_o, B_o, A_d, B_d


@pytest.mark.parametrize("name,N,K", [("gate_up", 2 * INTER, HIDDEN), ("down", HIDDEN, INTER)])
def test_qwen3_moe_grouped_full_size_sampled(routing, name, N, K):
    loads, off = routing
    T = int(off[-1])
    A_o, B_o, A_d, B_d = _operands(T, N, K, seed=7000 + K)
    rng = np.random.default_rng(N + K)
    rows = _sample_rows(loads, off, rng, 256, 8)
    cols = stratified(N, 128, rng, extra=(N - 8,))
    y_ref, yabs = par_grouped_gemm(orc, off, T, N, K, A_o, B_o, rows, cols)
    y = fp8.fp8_grouped_block_gemm(dev(off), A_d, B_d, T, N, K, fp8.OUT_BF16)
    fp8.device_status()
    yb = host(y)[np.ix_(rows, cols)]
    bad = orc.check_bf16(yb, y_ref, yabs, REL)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{name}: {int(bad.sum())}/{bad.size} outside tolerance; first "
                             f"(row {rows[i[0]]}, col {cols[i[1]]}): ref {y_ref[i]}")


def test_qwen3_moe_fused_swiglu_full_size_sampled(routing):
    loads, off = routing
    T = int(off[-1])
    N, K = 2 * INTER, HIDDEN
    A_o, B_o, A_d, B_d = _operands(T, N, K, seed=7100)
    rng = np.random.default_rng(11)
    rows = _sample_rows(loads, off, rng, 32, 2)
    y_ref, yabs = par_grouped_gemm(orc, off, T, N, K, A_o, B_o, rows, np.arange(N))
    tol = REL * yabs
    lo, hi = orc.swiglu_bounds(y_ref[:, :INTER], tol[:, :INTER], y_ref[:, INTER:], tol[:, INTER:])
    q, s = fp8.fp8_grouped_block_gemm_quant(dev(off), A_d, B_d, T, N, K, fp8.EPI_SWIGLU)
    fp8.device_status()
    bs, bc = orc.check_quantized_1x128(host(q)[rows], np.ascontiguousarray(host(s)[:, rows]), lo, hi,
                                       orc.E4M3, orc.SCALE_FP32)
    assert not bs.any() and not bc.any(), f"{int(bs.sum())} scales, {int(bc.sum())} codes rejected"
