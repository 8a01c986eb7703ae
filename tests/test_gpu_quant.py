"""Parity of the CUDA quantizers with the oracle: codes and scales bit-exact."""
import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import dev_bf16, f32_bits, host

pytestmark = pytest.mark.gpu


def _edge_cases(x: np.ndarray, seed: int) -> np.ndarray:
    """Plant the degenerate values the method has into a bf16 matrix."""
    x = x.copy()
    rng = np.random.default_rng(seed)
    M, K = x.shape
    x[0, :128] = 0                                     # all-zero tile
    x[min(1, M - 1), 0] = 0x8000                       # -0
    if M > 2:
        x[2, :128] = rng.integers(1, 0x80, 128).astype(np.uint16)      # bf16 subnormal tile
        x[2, 5] |= 0x8000
    if M > 3:
        x[3, 128 % K:128 % K + 128] = inputs.bf16_bits(np.full(128, 448.0, np.float32))  # exact fmax
    if M > 4 and K >= 256:
        x[4, 128:256] = inputs.bf16_bits(np.linspace(-3e38, 3e38, 128).astype(np.float32))  # huge
    if M > 5:
        x[5, :128] = inputs.bf16_bits((2.0 ** rng.integers(-30, 30, 128)).astype(np.float32))
    return x


SHAPES = [(1, 128), (5, 256), (37, 384), (256, 512), (129, 1024), (300, 640)]


@pytest.mark.parametrize("mode", [fp8.SCALE_FP32, fp8.SCALE_POW2])
@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
@pytest.mark.parametrize("M,K", SHAPES)
def test_quantize_1x128_parity(M, K, fmt, mode):
    x = _edge_cases(inputs.activations(M, K, seed=M + K), seed=1)
    q_ref, s_ref = orc.quantize_1x128(x, fmt, mode)
    q, s = fp8.fp8_quantize_1x128(dev_bf16(x), fmt, mode)
    assert np.array_equal(host(q), q_ref)
    assert np.array_equal(f32_bits(host(s)), f32_bits(s_ref))


@pytest.mark.parametrize("mode", [fp8.SCALE_FP32, fp8.SCALE_POW2])
@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
@pytest.mark.parametrize("N,K", [(1, 128), (100, 256), (128, 128), (300, 384), (513, 512)])
def test_quantize_128x128_parity(N, K, fmt, mode):
    w = _edge_cases(inputs.gaussian((N, K), 0.02, seed=N * K), seed=2)
    q_ref, s_ref = orc.quantize_128x128(w, fmt, mode)
    q, s = fp8.fp8_quantize_128x128(dev_bf16(w), fmt, mode)
    assert np.array_equal(host(q), q_ref)
    assert np.array_equal(f32_bits(host(s)), f32_bits(s_ref))


def test_quantize_strided_rows():
    """Row pitches larger than the row (a column slice of a wider matrix)."""
    import torch
    x = inputs.activations(64, 1024, seed=3)
    xd = dev_bf16(x)[:, 256:768]
    q = torch.empty((64, 1024), dtype=torch.uint8, device="cuda")[:, 128:640]
    q_ref, s_ref = orc.quantize_1x128(np.ascontiguousarray(x[:, 256:768]))
    q, s = fp8.fp8_quantize_1x128(xd, q=q)
    assert np.array_equal(host(q), q_ref) and np.array_equal(host(s), s_ref)


@pytest.mark.parametrize("fmt,mode", [(fp8.E4M3, fp8.SCALE_POW2), (fp8.E4M3, fp8.SCALE_FP32)])
def test_quantize_full_size(fmt, mode):
    """Largest activation and weight of the Llama-3.1-8B-shaped linears."""
    x = inputs.activations(8192, 14336, seed=21)
    q_ref, s_ref = orc.quantize_1x128(x, fmt, mode)
    q, s = fp8.fp8_quantize_1x128(dev_bf16(x), fmt, mode)
    assert np.array_equal(host(q), q_ref) and np.array_equal(f32_bits(host(s)), f32_bits(s_ref))
    del x, q_ref, s_ref, q, s
    w = inputs.gaussian((28672, 4096), 0.02, seed=22)
    q_ref, s_ref = orc.quantize_128x128(w, fmt, mode)
    q, s = fp8.fp8_quantize_128x128(dev_bf16(w), fmt, mode)
    assert np.array_equal(host(q), q_ref) and np.array_equal(f32_bits(host(s)), f32_bits(s_ref))


def test_pow2_scales_are_ue8m0_exact():
    """pow2 scales are exact powers of two (mantissa 0), as the MX path needs."""
    x = inputs.activations(256, 1024, seed=4)
    _, s = fp8.fp8_quantize_1x128(dev_bf16(x), fp8.E4M3, fp8.SCALE_POW2)
    assert np.all((f32_bits(host(s)) & 0x7FFFFF) == 0)


@pytest.mark.parametrize("M,N,K", [(300, 520, 640), (8192, 6144, 4096), (1, 128, 128), (0, 256, 256),
                                   (256, 0, 256)])
@pytest.mark.parametrize("fmt,mode", [(fp8.E4M3, fp8.SCALE_FP32), (fp8.E5M2, fp8.SCALE_POW2)])
def test_quantize_linear_equals_the_two_quantizers(M, N, K, fmt, mode):
    """One launch for a linear's X (1x128) and W (128x128): bit-exact with the
    oracle (ragged rows of both, full Llama-3.1-8B QKV size, empty operands)."""
    import torch
    x = inputs.activations(M, K, seed=M + 1)
    w = inputs.gaussian((N, K), 0.02, seed=N + 2)
    qx, sx, qw, sw = fp8.fp8_quantize_linear(dev_bf16(x) if M else torch.empty((0, K), dtype=torch.bfloat16,
                                                                               device="cuda"),
                                             dev_bf16(w) if N else torch.empty((0, K), dtype=torch.bfloat16,
                                                                               device="cuda"), fmt, mode)
    if M:
        rq, rs = orc.quantize_1x128(x, fmt, mode)
        assert np.array_equal(host(qx), rq) and np.array_equal(f32_bits(host(sx)), f32_bits(rs))
    if N:
        rq, rs = orc.quantize_128x128(w, fmt, mode)
        assert np.array_equal(host(qw), rq) and np.array_equal(f32_bits(host(sw)), f32_bits(rs))
