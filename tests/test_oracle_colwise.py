"""Pins of the oracle pieces behind the block-scaled backward pass: the
column-wise (transposed) 1x128 quantizer and products whose B operand has
one scale per 128 K-elements of each column.  References: numpy tile
reductions along columns with a brute-force nearest-code search, and numpy's
fp64 matmul of the dequantized operands."""
import numpy as np
import pytest
import torch

import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from test_oracle_fused import _nearest_code


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_colwise_tiles_match_numpy_and_brute_force(fmt):
    rows, cols = 384, 200                     # a partial last column block is fine for the oracle
    x = inputs.activations(rows, cols, seed=21)
    x[130, 17] = inputs.bf16_bits(np.float32([-3000.0]))[0]   # a block maximum mid-column
    xf = inputs.bits_to_f32(x)
    qt, st = orc.quantize_1x128_colwise(x, fmt, orc.SCALE_FP32)
    assert qt.shape == (cols, rows) and st.shape == (rows // 128, cols)
    amax = np.abs(xf).reshape(rows // 128, 128, cols).max(axis=1)          # [rows/128, cols]
    fm = np.float32(448.0 if fmt == orc.E4M3 else 57344.0)
    want = np.maximum((amax / fm).astype(np.float32), np.float32(2.0 ** -126))
    want = np.where(amax == 0, np.float32(1.0), want)
    assert np.array_equal(st, want)
    r = (np.float32(1.0) / np.repeat(want, 128, axis=0)).astype(np.float32)  # [rows, cols]
    assert np.array_equal(qt, _nearest_code((xf * r).astype(np.float32), fmt).T)


def test_gemm_with_per_column_b_scales_matches_numpy():
    M, N, K = 20, 40, 384
    qa, sa = orc.quantize_1x128(inputs.activations(M, K, seed=22))
    qb, sb = orc.quantize_1x128(inputs.activations(N, K, seed=23))
    y, ya = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa),
                     orc.operand(qb, orc.E4M3, orc.GRAN_1x128, sb))
    dec = lambda q: torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    A = dec(qa) * np.repeat(sa.T.astype(np.float64), 128, axis=1)
    B = dec(qb) * np.repeat(sb.T.astype(np.float64), 128, axis=1)
    ref = A @ B.T
    assert np.all(np.abs(y - ref) <= 1e-12 * (np.abs(A) @ np.abs(B).T))
    assert np.allclose(ya, np.abs(A) @ np.abs(B).T, rtol=1e-12, atol=0)


def test_wgrad_of_colwise_copies_is_the_transposed_product():
    """dW = dY^T X from the column-wise copies equals the product of the
    dequantized column-wise tiles of dY and X (numpy), i.e. the contraction
    runs over the tokens with one scale per 128 tokens per column."""
    M, n_out, k_in = 256, 24, 16
    dy = inputs.student_t((M, n_out), 3.0, 1e-3, seed=24)
    x = inputs.activations(M, k_in, seed=25)
    qdt, sdt = orc.quantize_1x128_colwise(dy)
    qxt, sxt = orc.quantize_1x128_colwise(x)
    y, _ = orc.gemm(n_out, k_in, M, orc.operand(qdt, orc.E4M3, orc.GRAN_1x128, sdt),
                    orc.operand(qxt, orc.E4M3, orc.GRAN_1x128, sxt))
    dec = lambda q: torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    dY = dec(qdt.T) * np.repeat(sdt.astype(np.float64), 128, axis=0)     # [M, n_out]
    X = dec(qxt.T) * np.repeat(sxt.astype(np.float64), 128, axis=0)      # [M, k_in]
    ref = dY.T @ X
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-300)
