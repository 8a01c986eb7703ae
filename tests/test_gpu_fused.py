"""Parity of the quantized-output product (fp8_block_gemm_quant and its
grouped form) with the oracle.

The kernel quantizes its own fp32 result, which matches the oracle's exact
(fp64) sum only within the product tolerance |y - y_ref| <= 1e-5 sum|terms|.
So codes and scales are accepted when they are the 1x128 quantization of
SOME fp32 values inside that tolerance (oracle.check_quantized_1x128); with
SwiGLU, of some value of silu(gate) * up over the gate and up tolerances
(oracle.swiglu_bounds).  Where the product is exact in fp32 (small integer
inputs, unit scales) the codes and scales must equal the oracle's
quantization of the exact result bit for bit."""
import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import dev, host, stratified

pytestmark = pytest.mark.gpu
REL = 1e-5


def _operands(M, N, K, mode, seed, w=None):
    x = inputs.activations(M, K, seed=seed)
    w = inputs.gaussian((N, K), 0.02, seed=seed + 1) if w is None else w
    qa, sa = orc.quantize_1x128(x, orc.E4M3, mode)
    qb, sb = orc.quantize_128x128(w, orc.E4M3, mode)
    A_o = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B_o = orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb)
    A_d = fp8.operand(dev(qa), dev(sa))
    B_d = fp8.operand(dev(qb), dev(sb), gran=fp8.GRAN_128x128)
    return A_o, B_o, A_d, B_d


def _assert_accepted(q, s, lo, hi, q_fmt, q_mode, what=""):
    bs, bc = orc.check_quantized_1x128(q, s, lo, hi, q_fmt, q_mode)
    if bs.any() or bc.any():
        msg = f"{what}: {int(bs.sum())} scales, {int(bc.sum())} codes rejected"
        if bc.any():
            i = tuple(np.argwhere(bc)[0])
            msg += f"; first code {i}: got 0x{int(q[i]):02x} interval [{lo[i]}, {hi[i]}]"
        if bs.any():
            j = tuple(np.argwhere(bs)[0])
            msg += f"; first scale {j}: got {s[j]}"
        raise AssertionError(msg)


@pytest.mark.parametrize("mode", [fp8.SCALE_FP32, fp8.SCALE_POW2], ids=["promote", "mx"])
@pytest.mark.parametrize("q_fmt,q_mode", [(fp8.E4M3, fp8.SCALE_FP32), (fp8.E4M3, fp8.SCALE_POW2),
                                          (fp8.E5M2, fp8.SCALE_FP32)], ids=["e4m3", "e4m3pow2", "e5m2"])
def test_quantized_output(mode, q_fmt, q_mode):
    # ragged M, N of 2.5 tiles (the last tile's second half is past N), 3 K blocks
    M, N, K = 300, 640, 384
    A_o, B_o, A_d, B_d = _operands(M, N, K, mode, seed=51)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    q, s = fp8.fp8_block_gemm_quant(A_d, B_d, M, N, K, fp8.EPI_NONE, q_fmt, q_mode, mode)
    tol = REL * yabs
    _assert_accepted(host(q), host(s), y_ref - tol, y_ref + tol, q_fmt, q_mode)
    fp8.device_status()


@pytest.mark.parametrize("mode", [fp8.SCALE_FP32, fp8.SCALE_POW2], ids=["promote", "mx"])
@pytest.mark.parametrize("q_mode", [fp8.SCALE_FP32, fp8.SCALE_POW2])
def test_quantized_output_exact_case_is_bit_exact(mode, q_mode):
    """Integer-valued E4M3 inputs (|v| <= 8) with unit scales and K = 256: every
    fp32 partial sum is exact, so the kernel quantizes exactly y_ref."""
    M, N, K = 256, 512, 256
    rng = np.random.default_rng(61)
    ia = rng.integers(-8, 9, (M, K)).astype(np.float32)
    ib = rng.integers(-8, 9, (N, K)).astype(np.float32)
    ia[5, :] = 0.0                                    # a zero output row: scale 1, codes 0
    qa, qb = orc.encode_array(ia, orc.E4M3), orc.encode_array(ib, orc.E4M3)
    sa = np.ones((K // 128, M), np.float32)
    sb = np.ones((N // 128, K // 128), np.float32)
    y_ref, _ = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa),
                        orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb))
    y32 = y_ref.astype(np.float32)
    assert np.array_equal(y32.astype(np.float64), y_ref)
    q_ref, s_ref = orc.quantize_1x128_f32(y32, orc.E4M3, q_mode)
    q, s = fp8.fp8_block_gemm_quant(fp8.operand(dev(qa), dev(sa)),
                                    fp8.operand(dev(qb), dev(sb), gran=fp8.GRAN_128x128),
                                    M, N, K, fp8.EPI_NONE, fp8.E4M3, q_mode, mode)
    assert np.array_equal(host(s), s_ref)
    assert np.array_equal(host(q), q_ref)


def _swiglu_interval(y_ref, yabs, I):
    g, u = y_ref[:, :I], y_ref[:, I:]
    return orc.swiglu_bounds(g, REL * yabs[:, :I], u, REL * yabs[:, I:])


@pytest.mark.parametrize("mode", [fp8.SCALE_FP32, fp8.SCALE_POW2], ids=["promote", "mx"])
@pytest.mark.parametrize("q_mode", [fp8.SCALE_FP32, fp8.SCALE_POW2])
def test_swiglu_output(mode, q_mode):
    M, I, K = 300, 384, 512
    N = 2 * I
    A_o, B_o, A_d, B_d = _operands(M, N, K, mode, seed=71)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    lo, hi = _swiglu_interval(y_ref, yabs, I)
    q, s = fp8.fp8_block_gemm_quant(A_d, B_d, M, N, K, fp8.EPI_SWIGLU, fp8.E4M3, q_mode, mode)
    assert tuple(q.shape) == (M, I) and tuple(s.shape) == (I // 128, M)
    _assert_accepted(host(q), host(s), lo, hi, fp8.E4M3, q_mode)
    fp8.device_status()


def test_grouped_swiglu_output():
    import torch
    G, I, K = 5, 256, 256
    N = 2 * I
    loads = np.array([130, 0, 260, 10, 1])            # an empty group and a one-row group
    off = np.zeros(G + 1, np.int32)
    off[1:] = np.cumsum(loads)
    T = int(off[-1])
    a_rows = T + 7                                    # rows past the last group: untouched
    x = inputs.activations(a_rows, K, seed=81)
    w = inputs.gaussian((G * N, K), 0.02, seed=82)
    qa, sa = orc.quantize_1x128(x)
    qw = np.empty((G * N, K), np.uint8)
    sw = np.empty((G, N // 128, K // 128), np.float32)
    for g in range(G):
        qw[g * N:(g + 1) * N], sw[g] = orc.quantize_128x128(w[g * N:(g + 1) * N])
    A_o = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B_o = orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw)
    y_ref, yabs = orc.grouped_gemm(off, a_rows, N, K, A_o, B_o, rows=np.arange(T))
    lo, hi = _swiglu_interval(y_ref, yabs, I)
    q = torch.full((a_rows, I), 0x5A, dtype=torch.uint8, device="cuda")
    s = torch.full((I // 128, a_rows), float("nan"), device="cuda")
    fp8.fp8_grouped_block_gemm_quant(dev(off), fp8.operand(dev(qa), dev(sa)),
                                     fp8.operand(dev(qw), dev(sw), gran=fp8.GRAN_128x128),
                                     a_rows, N, K, fp8.EPI_SWIGLU, q=q, q_scales=s)
    qh, sh = host(q), host(s)
    _assert_accepted(qh[:T], sh[:, :T], lo, hi, fp8.E4M3, fp8.SCALE_FP32)
    assert np.all(qh[T:] == 0x5A) and np.all(np.isnan(sh[:, T:]))


def test_grouped_quantized_output_plain():
    G, N, K = 3, 384, 384
    loads = np.array([200, 57, 0])
    off = np.zeros(G + 1, np.int32)
    off[1:] = np.cumsum(loads)
    T = int(off[-1])
    x = inputs.activations(T, K, seed=91)
    w = inputs.gaussian((G * N, K), 0.02, seed=92)
    qa, sa = orc.quantize_1x128(x)
    qw = np.empty((G * N, K), np.uint8)
    sw = np.empty((G, N // 128, K // 128), np.float32)
    for g in range(G):
        qw[g * N:(g + 1) * N], sw[g] = orc.quantize_128x128(w[g * N:(g + 1) * N])
    y_ref, yabs = orc.grouped_gemm(off, T, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa),
                                   orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw))
    q, s = fp8.fp8_grouped_block_gemm_quant(dev(off), fp8.operand(dev(qa), dev(sa)),
                                            fp8.operand(dev(qw), dev(sw), gran=fp8.GRAN_128x128),
                                            T, N, K, fp8.EPI_NONE)
    tol = REL * yabs
    _assert_accepted(host(q), host(s), y_ref - tol, y_ref + tol, fp8.E4M3, fp8.SCALE_FP32)


def test_empty_contraction_gives_zero_codes_and_unit_scales():
    import torch
    M, N = 130, 256
    A_d = fp8.operand(torch.zeros((M, 16), dtype=torch.uint8, device="cuda"),
                      torch.ones((1, M), device="cuda"))
    B_d = fp8.operand(torch.zeros((N, 16), dtype=torch.uint8, device="cuda"),
                      torch.ones((2, 1), device="cuda"), gran=fp8.GRAN_128x128)
    q, s = fp8.fp8_block_gemm_quant(A_d, B_d, M, N, 0, fp8.EPI_SWIGLU)
    assert np.all(host(q) == 0) and np.all(host(s) == 1.0)


def test_llama31_8b_gate_up_swiglu_sampled():
    """The Llama-3.1-8B MLP's gate/up product (M = 8192, 2 x 14336 rows) with
    SwiGLU and quantization to the down product's operand, at full size, in
    the configuration the benchmark times; checked on sampled rows and on
    sampled 128-column output blocks."""
    M, I, K = 8192, 14336, 4096
    N = 2 * I
    x = inputs.activations(M, K, seed=1000 + K)
    w = inputs.gaussian((N, K), 0.02, seed=2000 + N)
    qa, sa = orc.quantize_1x128(x)
    qb, sb = orc.quantize_128x128(w)
    rng = np.random.default_rng(5)
    rows = stratified(M, 256, rng)
    blocks = np.unique(np.concatenate([[0, I // 128 - 1], rng.integers(0, I // 128, 4)]))
    hcols = (blocks[:, None] * 128 + np.arange(128)[None, :]).ravel()
    cols = np.concatenate([hcols, I + hcols])
    y_ref, yabs = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa),
                           orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb), rows=rows, cols=cols)
    lo, hi = _swiglu_interval(y_ref, yabs, hcols.size)
    q, s = fp8.fp8_block_gemm_quant(fp8.operand(dev(qa), dev(sa)),
                                    fp8.operand(dev(qb), dev(sb), gran=fp8.GRAN_128x128),
                                    M, N, K, fp8.EPI_SWIGLU)
    qh, sh = host(q), host(s)
    _assert_accepted(qh[np.ix_(rows, hcols)], sh[np.ix_(blocks, rows)], lo, hi, fp8.E4M3,
                     fp8.SCALE_FP32)
