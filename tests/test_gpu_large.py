"""Operands beyond 2^31 elements / bytes: the quantizers and the promotion
product index past the 32-bit range.  The large tensors repeat a seeded block
whose row count (250, 3000) does not divide the 2^31 boundary, so an index
that wrapped at 32 bits would land on a different row of the block; every
sampled row is compared with the oracle run on the block rows it repeats."""
import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import dev, dev_bf16, f32_bits, host, par_gemm, par_quantize_1x128, stratified

pytestmark = pytest.mark.gpu


def test_quantizers_beyond_2_31_elements():
    import torch
    P, K, reps = 250, 131072, 67                      # 16750 x 131072 = 2.195e9 elements
    rows = P * reps
    assert rows * K > 2 ** 31 and (2 ** 31 // K) % P != 0
    blk = inputs.activations(P, K, seed=31)
    x = dev_bf16(blk).repeat(reps, 1)
    assert x.shape == (rows, K)

    # 1x128: rows around element 2^31 (row 16384) and at the end
    q_ref, s_ref = par_quantize_1x128(orc, blk, orc.E4M3, orc.SCALE_FP32)
    q, s = fp8.fp8_quantize_1x128(x)
    check = [16382, 16383, 16384, 16385, 2 ** 31 // K + 200, rows - 2, rows - 1]
    idx = torch.tensor(check, device=x.device)
    q_rows = host(q.index_select(0, idx))
    s_cols = host(s.index_select(1, idx))
    for i, r in enumerate(check):
        assert np.array_equal(q_rows[i], q_ref[r % P]), r
        assert np.array_equal(f32_bits(s_cols[:, i]), f32_bits(s_ref[:, r % P])), r
    del q, s

    # 128x128: the row band that holds element 2^31 and the partial last band
    q, s = fp8.fp8_quantize_128x128(x)
    for b0 in (16384, (rows // 128) * 128):
        b1 = min(b0 + 128, rows)
        band = blk[np.arange(b0, b1) % P]
        qb_ref, sb_ref = orc.quantize_128x128(band)
        assert np.array_equal(host(q[b0:b1]), qb_ref), b0
        assert np.array_equal(f32_bits(host(s[b0 // 128])), f32_bits(sb_ref[0])), b0


@pytest.mark.parametrize("out", [fp8.OUT_F32, fp8.OUT_BF16], ids=["f32", "bf16"])
def test_gemm_a_beyond_2_31_bytes(out):
    """A [141000 x 16384] E4M3 (2.31e9 bytes) with 1x128 scales against one
    256-column block of W: rows before, at and after byte 2^31 (row 131072)
    and the last rows, every column."""
    import torch
    P, K, reps, N = 3000, 16384, 47, 256
    M = P * reps
    assert M * K > 2 ** 31 and (2 ** 31 // K) % P != 0
    a = inputs.activations(P, K, seed=41)
    w = inputs.gaussian((N, K), 0.02, seed=42)
    qa, sa = par_quantize_1x128(orc, a, orc.E4M3, orc.SCALE_FP32)
    qb, sb = orc.quantize_128x128(w)
    A_d = fp8.operand(dev(qa).repeat(reps, 1), dev(sa).repeat(1, reps))
    B_d = fp8.operand(dev(qb), dev(sb), gran=fp8.GRAN_128x128)
    y = fp8.fp8_block_gemm(A_d, B_d, M, N, K, out)
    rng = np.random.default_rng(43)
    dev_rows = np.unique(np.concatenate([
        np.array([131070, 131071, 131072, 131073, 131199, M - 129, M - 128, M - 1]),
        M - P + stratified(P, 256, rng)]))
    cols = np.arange(N)
    y_ref, yabs = par_gemm(orc, P, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa),
                           orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb), dev_rows % P, cols)
    yd = host(y.index_select(0, torch.tensor(dev_rows, device=y.device)))
    if out == fp8.OUT_F32:
        bad = orc.check_f32(yd, y_ref, yabs)
    else:
        bad = orc.check_bf16(yd.view(np.uint16), y_ref, yabs)
    assert int(bad.sum()) == 0, f"{int(bad.sum())}/{bad.size} outside tolerance"
