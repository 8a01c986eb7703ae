"""Parity of the block-scaled backward pass with the oracle: the column-wise
(transposed) 1x128 quantizer, bit for bit, and the products whose B operand
has one scale per 128 K-elements of each column (1x128 B), checked with the
product tolerance |y - y_ref| <= 1e-5 sum|terms|."""
import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import dev, dev_bf16, host, stratified

pytestmark = pytest.mark.gpu
REL = 1e-5


@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
@pytest.mark.parametrize("mode", [fp8.SCALE_FP32, fp8.SCALE_POW2])
@pytest.mark.parametrize("rowwise", [False, True])
def test_colwise_quantizer_bit_exact(fmt, mode, rowwise):
    rows, cols = 384, 640
    x = inputs.activations(rows, cols, seed=101)
    x[7 * 16: 8 * 16, 128:256] = 0                      # part of a column block is zero
    x[256:384, 512:640] = 0                             # a whole zero tile: scales 1
    qt_ref, st_ref = orc.quantize_1x128_colwise(x, fmt, mode)
    out = fp8.fp8_quantize_1x128_colwise(dev_bf16(x), fmt, mode, rowwise=rowwise)
    assert np.array_equal(host(out[1]), st_ref)
    assert np.array_equal(host(out[0]), qt_ref)
    if rowwise:
        q_ref, s_ref = orc.quantize_1x128(x, fmt, mode)
        assert np.array_equal(host(out[3]), s_ref)
        assert np.array_equal(host(out[2]), q_ref)


def test_colwise_quantizer_full_size_gradient():
    """dY of the Llama-3.1-8B up-projection backward ([8192, 14336], heavy
    tails), both copies, every byte and scale."""
    rows, cols = 8192, 14336
    dy = inputs.student_t((rows, cols), 3.0, 1e-3, seed=100)
    qt_ref, st_ref = orc.quantize_1x128_colwise(dy)
    q_ref, s_ref = orc.quantize_1x128(dy)
    qt, st, q, s = fp8.fp8_quantize_1x128_colwise(dev_bf16(dy), rowwise=True)
    assert np.array_equal(host(st), st_ref) and np.array_equal(host(s), s_ref)
    assert np.array_equal(host(qt), qt_ref) and np.array_equal(host(q), q_ref)


def test_colwise_quantizer_padded_leading_dimensions():
    import torch
    rows, cols = 256, 384
    x = inputs.activations(rows, cols, seed=103)
    xd = torch.zeros((rows, cols + 64), dtype=torch.bfloat16, device="cuda")
    xd[:, :cols] = dev_bf16(x)
    qt = torch.full((cols, rows + 32), 0x77, dtype=torch.uint8, device="cuda")
    st = torch.empty((rows // 128, cols), device="cuda")
    fp8.fp8_quantize_1x128_colwise(xd[:, :cols], qt=qt[:, :rows], scales_t=st)
    qt_ref, st_ref = orc.quantize_1x128_colwise(x)
    qh = host(qt)
    assert np.array_equal(qh[:, :rows], qt_ref) and np.all(qh[:, rows:] == 0x77)
    assert np.array_equal(host(st), st_ref)


def _col_operands(M, N, K, seed, fa=orc.E4M3, fb=orc.E4M3, mode=orc.SCALE_FP32, a_gran=orc.GRAN_1x128):
    a = inputs.activations(M, K, seed=seed)
    b = inputs.activations(N, K, seed=seed + 1)
    qa, sa = (orc.quantize_1x128(a, fa, mode) if a_gran == orc.GRAN_1x128
              else orc.quantize_128x128(a, fa, mode))
    qb, sb = orc.quantize_1x128(b, fb, mode)           # B: one scale per 128 K of each column
    A_o = orc.operand(qa, fa, a_gran, sa)
    B_o = orc.operand(qb, fb, orc.GRAN_1x128, sb)
    A_d = fp8.operand(dev(qa), dev(sa), fa, a_gran)
    B_d = fp8.operand(dev(qb), dev(sb), fb, fp8.GRAN_1x128)
    return A_o, B_o, A_d, B_d


def _check(y, y_ref, yabs, out):
    if out == fp8.OUT_F32:
        bad = orc.check_f32(y, y_ref, yabs, REL)
    else:
        bad = orc.check_bf16(y.view(np.uint16), y_ref, yabs, REL)
    assert not bad.any(), f"{int(bad.sum())}/{bad.size} outside tolerance"


@pytest.mark.parametrize("M,N,K", [(300, 384, 512), (128, 136, 128), (640, 1024, 1152)])
@pytest.mark.parametrize("out", [fp8.OUT_F32, fp8.OUT_BF16])
def test_gemm_with_per_column_b_scales(M, N, K, out):
    A_o, B_o, A_d, B_d = _col_operands(M, N, K, seed=111)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    _check(host(fp8.fp8_block_gemm(A_d, B_d, M, N, K, out)), y_ref, yabs, out)


@pytest.mark.parametrize("mode", [fp8.SCALE_FP32, fp8.SCALE_POW2])
def test_gemm_per_column_b_modes_formats_and_a_granularities(mode):
    M, N, K = 256, 512, 384
    for fa, fb, ag in ((orc.E5M2, orc.E4M3, orc.GRAN_1x128), (orc.E4M3, orc.E5M2, orc.GRAN_128x128)):
        A_o, B_o, A_d, B_d = _col_operands(M, N, K, seed=121, fa=fa, fb=fb, mode=mode, a_gran=ag)
        y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
        _check(host(fp8.fp8_block_gemm(A_d, B_d, M, N, K, fp8.OUT_F32, mode)), y_ref, yabs, fp8.OUT_F32)


def test_wgrad_from_colwise_copies():
    """dW = dY^T X with both operands from the column-wise quantizer (GPU),
    against the oracle product of the oracle's column-wise copies."""
    M, n_out, k_in = 512, 384, 256
    dy = inputs.student_t((M, n_out), 3.0, 1e-3, seed=131)
    x = inputs.activations(M, k_in, seed=132)
    qdt, sdt = orc.quantize_1x128_colwise(dy)
    qxt, sxt = orc.quantize_1x128_colwise(x)
    y_ref, yabs = orc.gemm(n_out, k_in, M, orc.operand(qdt, orc.E4M3, orc.GRAN_1x128, sdt),
                           orc.operand(qxt, orc.E4M3, orc.GRAN_1x128, sxt))
    gq_dt, gs_dt = fp8.fp8_quantize_1x128_colwise(dev_bf16(dy))
    gq_xt, gs_xt = fp8.fp8_quantize_1x128_colwise(dev_bf16(x))
    dw = fp8.fp8_block_gemm(fp8.operand(gq_dt, gs_dt), fp8.operand(gq_xt, gs_xt, gran=fp8.GRAN_1x128),
                            n_out, k_in, M, fp8.OUT_F32)
    _check(host(dw), y_ref, yabs, fp8.OUT_F32)


@pytest.mark.parametrize("n_out,k_in", [(14336, 4096), (4096, 14336)], ids=["up", "down"])
def test_llama31_8b_wgrad_blockwise_sampled(n_out, k_in):
    """Full-size Llama-3.1-8B MLP wgrad products of the block recipe (M = 8192
    tokens contracted), sampled outputs."""
    M = 8192
    dy = inputs.student_t((M, n_out), 3.0, 1e-3, seed=100 + n_out)
    x = inputs.activations(M, k_in, seed=200 + k_in)
    qdt, sdt = orc.quantize_1x128_colwise(dy)
    qxt, sxt = orc.quantize_1x128_colwise(x)
    rng = np.random.default_rng(n_out)
    rows, cols = stratified(n_out, 256, rng), stratified(k_in, 256, rng, extra=(k_in - 8,))
    y_ref, yabs = orc.gemm(n_out, k_in, M, orc.operand(qdt, orc.E4M3, orc.GRAN_1x128, sdt),
                           orc.operand(qxt, orc.E4M3, orc.GRAN_1x128, sxt), rows=rows, cols=cols)
    dw = fp8.fp8_block_gemm(fp8.operand(dev(qdt), dev(sdt)),
                            fp8.operand(dev(qxt), dev(sxt), gran=fp8.GRAN_1x128), n_out, k_in, M, fp8.OUT_F32)
    _check(host(dw)[np.ix_(rows, cols)], y_ref, yabs, fp8.OUT_F32)
    fp8.device_status()
