"""Parity of the MXFP8 path with the oracle: the 1x32 quantizer (E8M0 scales,
floor rule) bit for bit, and the block-scaled product that applies the
per-32 scales in the tensor core, within |y - y_ref| <= 1e-5 sum|terms|."""
import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import dev, dev_bf16, host, stratified

pytestmark = pytest.mark.gpu
REL = 1e-5


@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
def test_mx_quantizer_bit_exact(fmt):
    rows, cols = 300, 640
    x = inputs.activations(rows, cols, seed=141)
    x[3, 32:64] = 0                                         # zero block: code 0
    x[4, 0] = inputs.bf16_bits(np.float32([500.0]))[0]       # saturating block maximum
    x[5, 128:160] = inputs.bf16_bits(np.float32([1e-39] * 32))  # subnormal block: code 0
    q_ref, s_ref = orc.quantize_mx(x, fmt)
    q, s = fp8.fp8_quantize_mx(dev_bf16(x), fmt)
    assert np.array_equal(host(s), s_ref)
    assert np.array_equal(host(q), q_ref)


def test_mx_quantizer_full_size():
    x = inputs.activations(8192, 4096, seed=142)
    w = inputs.gaussian((6144, 4096), 0.02, seed=143)
    for a in (x, w):
        q_ref, s_ref = orc.quantize_mx(a)
        q, s = fp8.fp8_quantize_mx(dev_bf16(a))
        assert np.array_equal(host(s), s_ref) and np.array_equal(host(q), q_ref)


def _mx_operands(M, N, K, seed, fa=orc.E4M3, fb=orc.E4M3, spread=False):
    a = inputs.activations(M, K, seed=seed)
    b = inputs.gaussian((N, K), 0.02, seed=seed + 1)
    if spread:   # 32-element blocks of very different magnitude: each K slice needs its own scale byte
        f = inputs.bits_to_f32(a) * np.tile(np.repeat(2.0 ** (4 * np.arange(4)), 32), K // 128)[None, :]
        a = inputs.bf16_bits(f.astype(np.float32))
        g = inputs.bits_to_f32(b) * np.tile(np.repeat(2.0 ** (-3 * np.arange(4)), 32), K // 128)[None, :]
        b = inputs.bf16_bits(g.astype(np.float32))
    qa, sa = orc.quantize_mx(a, fa)
    qb, sb = orc.quantize_mx(b, fb)
    A_o = orc.operand(qa, fa, orc.GRAN_1x32, sa)
    B_o = orc.operand(qb, fb, orc.GRAN_1x32, sb)
    A_d = fp8.operand(dev(qa), dev(sa), fa, fp8.GRAN_1x32)
    B_d = fp8.operand(dev(qb), dev(sb), fb, fp8.GRAN_1x32)
    return A_o, B_o, A_d, B_d


def _check(y, y_ref, yabs, out):
    if out == fp8.OUT_F32:
        bad = orc.check_f32(y, y_ref, yabs, REL)
    else:
        bad = orc.check_bf16(y.view(np.uint16), y_ref, yabs, REL)
    assert not bad.any(), f"{int(bad.sum())}/{bad.size} outside tolerance"


@pytest.mark.parametrize("spread", [False, True], ids=["activations", "spread-blocks"])
@pytest.mark.parametrize("out", [fp8.OUT_F32, fp8.OUT_BF16])
def test_mx_gemm(spread, out):
    M, N, K = 304, 640, 512                                # rows % 4 == 0 for A's scale table
    A_o, B_o, A_d, B_d = _mx_operands(M, N, K, seed=151, spread=spread)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    _check(host(fp8.fp8_block_gemm(A_d, B_d, M, N, K, out, fp8.SCALE_POW2)), y_ref, yabs, out)


def test_mx_gemm_mixed_formats_and_long_k():
    M, N, K = 256, 256, 2176
    A_o, B_o, A_d, B_d = _mx_operands(M, N, K, seed=161, fa=orc.E5M2, fb=orc.E4M3)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    _check(host(fp8.fp8_block_gemm(A_d, B_d, M, N, K, fp8.OUT_F32, fp8.SCALE_POW2)), y_ref, yabs, fp8.OUT_F32)


def test_mx_gemm_quantized_output():
    M, N, K = 256, 384, 256
    A_o, B_o, A_d, B_d = _mx_operands(M, N, K, seed=171)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    q, s = fp8.fp8_block_gemm_quant(A_d, B_d, M, N, K, fp8.EPI_NONE, fp8.E4M3, fp8.SCALE_POW2,
                                    fp8.SCALE_POW2)
    tol = REL * yabs
    bs, bc = orc.check_quantized_1x128(host(q), host(s), y_ref - tol, y_ref + tol, orc.E4M3,
                                       orc.SCALE_POW2)
    assert not bs.any() and not bc.any()


def test_mx_llama31_8b_gate_up_sampled():
    """Llama-3.1-8B gate/up (M = 8192, N = 28672, K = 4096) in MXFP8 at full
    size, as the MXFP8 fprop benchmark runs it; sampled outputs."""
    M, N, K = 8192, 28672, 4096
    x = inputs.activations(M, K, seed=1000 + K)
    w = inputs.gaussian((N, K), 0.02, seed=2000 + N)
    qa, sa = orc.quantize_mx(x)
    qb, sb = orc.quantize_mx(w)
    rng = np.random.default_rng(9)
    rows, cols = stratified(M, 128, rng), stratified(N, 256, rng, extra=(N - 8,))
    y_ref, yabs = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x32, sa),
                           orc.operand(qb, orc.E4M3, orc.GRAN_1x32, sb), rows=rows, cols=cols)
    y = fp8.fp8_block_gemm(fp8.operand(dev(qa), dev(sa), gran=fp8.GRAN_1x32),
                           fp8.operand(dev(qb), dev(sb), gran=fp8.GRAN_1x32), M, N, K, fp8.OUT_BF16,
                           fp8.SCALE_POW2)
    _check(host(y)[np.ix_(rows, cols)], y_ref, yabs, fp8.OUT_BF16)
    fp8.device_status()
