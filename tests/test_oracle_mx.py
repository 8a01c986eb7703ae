"""Pins of the MXFP8 oracle pieces (32-element blocks, E8M0 power-of-two
scales with the floor rule, products with per-32 scales).  References: a
brute-force search for the scale exponent, numpy block reductions with the
brute-force nearest-code search, closed-form examples, and numpy's fp64
matmul of the dequantized operands."""
import numpy as np
import pytest
import torch

import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from test_oracle_fused import _nearest_code

EMAX = {orc.E4M3: 8, orc.E5M2: 15}


def _brute_exponent(amax, fmt):
    """Largest e in [-127, 127] with 2^(e + emax) <= amax (-127 if none)."""
    if amax == 0:
        return -127
    best = -127
    for e in range(-127, 128):
        if 2.0 ** (e + EMAX[fmt]) <= amax:
            best = e
    return best


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_scale_code_matches_brute_force(fmt):
    rng = np.random.default_rng(2)
    vals = np.concatenate([np.float32([0.0, 1.0, 448.0, 500.0, 2.0 ** -133, 2.0 ** -126, 3.0e38, 255.9,
                                       256.0, 57344.0, 65536.0]),
                           (10.0 ** rng.uniform(-40, 38, 300)).astype(np.float32)])
    for a in vals:
        assert orc.mx_scale_code(float(a), fmt) == _brute_exponent(float(a), fmt) + 127, a
    assert orc.mx_scale_code(float("inf"), fmt) == 255 and orc.mx_scale_code(float("nan"), fmt) == 255


def test_scale_closed_forms():
    # E4M3: amax 1 -> 2^-8 (1.0 becomes 256); amax in [448, 512) -> scale 1
    assert orc.mx_scale_code(1.0, orc.E4M3) == 127 - 8
    assert orc.mx_scale_code(448.0, orc.E4M3) == 127 and orc.mx_scale_code(511.0, orc.E4M3) == 127
    # E5M2: amax 1 -> 2^-15 (1.0 becomes 32768)
    assert orc.mx_scale_code(1.0, orc.E5M2) == 127 - 15


def test_floor_rule_saturates_the_top_of_the_binade():
    x = np.zeros((1, 128), np.float32)
    x[0, 0], x[0, 1], x[0, 2] = 500.0, 256.0, -300.0       # scale 1: 500 -> 448, -300 -> -288
    q, s = orc.quantize_mx(inputs.bf16_bits(x))
    assert s[0, 0, 0] == 127
    assert q[0, 0] == 0x7E and q[0, 1] == 0x78 and q[0, 2] == 0xF9


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_quantize_mx_matches_numpy_blocks_and_brute_force(fmt):
    rows, cols = 9, 384
    x = inputs.activations(rows, cols, seed=12)
    x[2, 32:64] = 0                                        # a zero block: code 0
    xf = inputs.bits_to_f32(x)
    q, s = orc.quantize_mx(x, fmt)
    amax = np.abs(xf).reshape(rows, cols // 32, 32).max(axis=2)
    e = np.vectorize(lambda a: _brute_exponent(float(a), fmt))(amax)
    codes = (e + 127).astype(np.uint8)                      # [rows, cols/32]
    want = codes.reshape(rows, cols // 128, 4).transpose(1, 0, 2)
    assert np.array_equal(s, want)
    mult = np.repeat(np.exp2(-e.astype(np.float64)), 32, axis=1).astype(np.float32)
    assert np.array_equal(q, _nearest_code((xf * mult).astype(np.float32), fmt))


def test_gemm_with_mx_scales_matches_numpy():
    M, N, K = 12, 20, 256
    qa, sa = orc.quantize_mx(inputs.activations(M, K, seed=13))
    qb, sb = orc.quantize_mx(inputs.gaussian((N, K), 0.02, seed=14), orc.E5M2)
    y, _ = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x32, sa),
                    orc.operand(qb, orc.E5M2, orc.GRAN_1x32, sb))

    def deq(q, s, tt):
        rows = q.shape[0]
        codes = s.transpose(1, 0, 2).reshape(rows, -1).astype(np.float64)   # [rows, K/32]
        return (torch.from_numpy(q).view(tt).to(torch.float64).numpy()
                * np.repeat(np.exp2(codes - 127), 32, axis=1))

    A = deq(qa, sa, torch.float8_e4m3fn)
    B = deq(qb, sb, torch.float8_e5m2)
    assert np.all(np.abs(y - A @ B.T) <= 1e-12 * (np.abs(A) @ np.abs(B).T))
