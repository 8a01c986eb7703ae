"""The threaded drivers of the oracle used by the full-size GPU tests and the
benchmark's CPU baseline split rows over host threads.  They must return
exactly what the single-threaded oracle returns."""
import numpy as np

import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import (par_gemm, par_grouped_gemm, par_quantize_1x128, par_quantize_128x128,
                     par_quantize_tensor)


def test_parallel_quantizers_equal_the_serial_oracle():
    x = inputs.activations(389, 512, seed=3)                 # rows not a multiple of the chunking
    for mode in (orc.SCALE_FP32, orc.SCALE_POW2):
        q1, s1 = orc.quantize_1x128(x, orc.E4M3, mode)
        q2, s2 = par_quantize_1x128(orc, x, orc.E4M3, mode)
        assert np.array_equal(q1, q2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
        q1, s1 = orc.quantize_128x128(x, orc.E5M2, mode)     # ragged last row-tile
        q2, s2 = par_quantize_128x128(orc, x, orc.E5M2, mode)
        assert np.array_equal(q1, q2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    q1, a1 = orc.quantize_tensor(x, orc.E5M2, 3e-3)
    q2, a2 = par_quantize_tensor(orc, x, orc.E5M2, 3e-3)
    assert np.array_equal(q1, q2) and np.float32(a1) == np.float32(a2)


def test_parallel_products_equal_the_serial_oracle():
    M, N, K = 300, 256, 384
    qa, sa = orc.quantize_1x128(inputs.activations(M, K, seed=5))
    qb, sb = orc.quantize_128x128(inputs.gaussian((2 * N, K), 0.02, seed=6))
    A = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B = orc.operand(qb[:N], orc.E4M3, orc.GRAN_128x128, sb[:N // 128])
    rows, cols = np.arange(0, M, 7), np.arange(0, N, 5)
    y1, a1 = orc.gemm(M, N, K, A, B, rows=rows, cols=cols)
    y2, a2 = par_gemm(orc, M, N, K, A, B, rows, cols)
    assert np.array_equal(y1, y2) and np.array_equal(a1, a2)
    off = np.array([0, 120, 300], np.int32)
    Bg = orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb.reshape(2, N // 128, K // 128))
    y1, a1 = orc.grouped_gemm(off, M, N, K, A, Bg, rows=rows, cols=cols)
    y2, a2 = par_grouped_gemm(orc, off, M, N, K, A, Bg, rows, cols)
    assert np.array_equal(y1, y2) and np.array_equal(a1, a2)
