"""Pins of the oracle's fp64 block-scaled GEMM and of the acceptance rules.

- numpy float64 matmul (a library routine) of operands dequantized through
  PyTorch's float8 decode and numpy scale expansion -- independent of the
  oracle's own decode and scale lookup;
- exact special cases: a scaled identity in one 128-block, integer-valued
  products whose sums are exact;
- storage transposition and the orientation of every scale table;
- the grouped product against per-group numpy matmuls, empty groups, rows
  outside every group.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs

TORCH_T = {orc.E4M3: torch.float8_e4m3fn, orc.E5M2: torch.float8_e5m2}


def _deq_codes(q, fmt):
    return torch.from_numpy(np.ascontiguousarray(q)).view(TORCH_T[fmt]).to(torch.float64).numpy()


def _expand(scales, gran, rows, K, transposed=False):
    """Scale of every logical element [rows, K] from a scale table."""
    if gran == orc.GRAN_TENSOR:
        return np.full((rows, K), float(scales.ravel()[0]))
    if gran == orc.GRAN_1x128:
        return np.repeat(scales.T.astype(np.float64), 128, axis=1)[:, :K]
    t = scales.T if transposed else scales
    return np.repeat(np.repeat(t.astype(np.float64), 128, axis=0), 128, axis=1)[:rows, :K]


def _numpy_ref(qa, sa, ga, fa, qb, sb, gb, fb, M, N, K, ta=False, tb=False):
    A = _deq_codes(qa.T if ta else qa, fa) * _expand(sa, ga, M, K, ta)
    B = _deq_codes(qb.T if tb else qb, fb) * _expand(sb, gb, N, K, tb)
    return A @ B.T, np.abs(A) @ np.abs(B).T


@pytest.mark.parametrize("fa,fb", [(orc.E4M3, orc.E4M3), (orc.E5M2, orc.E4M3)])
def test_gemm_vs_numpy_blockwise(fa, fb):
    M, N, K = 70, 260, 384
    x = inputs.activations(M, K, seed=0)
    w = inputs.gaussian((N, K), 0.02, seed=1)
    qa, sa = orc.quantize_1x128(x, fa, orc.SCALE_FP32)
    qb, sb = orc.quantize_128x128(w, fb, orc.SCALE_FP32)
    A = orc.operand(qa, fa, orc.GRAN_1x128, sa)
    B = orc.operand(qb, fb, orc.GRAN_128x128, sb)
    y, ya = orc.gemm(M, N, K, A, B)
    yr, yar = _numpy_ref(qa, sa, orc.GRAN_1x128, fa, qb, sb, orc.GRAN_128x128, fb, M, N, K)
    assert np.all(np.abs(y - yr) <= 1e-13 * yar)
    assert np.allclose(ya, yar, rtol=1e-13, atol=0)
    # selections return the same numbers as the full product
    rows, cols = np.array([0, 69, 33]), np.array([259, 0, 128, 127])
    ys, _ = orc.gemm(M, N, K, A, B, rows=rows, cols=cols)
    assert np.array_equal(ys, y[np.ix_(rows, cols)])


def test_gemm_transposed_storage_and_scale_orientation():
    M, N, K = 130, 256, 256
    a = inputs.gaussian((M, K), 1.0, seed=3)
    b = inputs.gaussian((N, K), 0.02, seed=4)
    qa, sa = orc.quantize_128x128(a, orc.E4M3, orc.SCALE_POW2)
    qb, sb = orc.quantize_128x128(b, orc.E4M3, orc.SCALE_FP32)
    y0, a0 = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_128x128, sa),
                      orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb))
    # the same matrices stored [K][rows] with scale tables in stored orientation
    y1, a1 = orc.gemm(M, N, K,
                      orc.operand(qa.T.copy(), orc.E4M3, orc.GRAN_128x128, sa.T.copy(), transposed=True),
                      orc.operand(qb.T.copy(), orc.E4M3, orc.GRAN_128x128, sb.T.copy(), transposed=True))
    assert np.array_equal(y0, y1) and np.array_equal(a0, a1)
    yr, _ = _numpy_ref(qa.T.copy(), sa.T.copy(), orc.GRAN_128x128, orc.E4M3,
                       qb.T.copy(), sb.T.copy(), orc.GRAN_128x128, orc.E4M3, M, N, K, ta=True, tb=True)
    assert np.all(np.abs(y0 - yr) <= 1e-13 * a0)


def test_gemm_per_tensor_mixed_formats():
    M, N, K = 64, 128, 512
    dy = inputs.student_t((M, K), 3.0, 1e-3, seed=100)
    w = inputs.gaussian((N, K), 0.02, seed=1)
    qa, _ = orc.quantize_tensor(dy, orc.E5M2, 3.0e-7)
    qb, _ = orc.quantize_tensor(w, orc.E4M3, 2.0e-4)
    sa, sb = np.float32([3.0e-7]), np.float32([2.0e-4])
    y, ya = orc.gemm(M, N, K, orc.operand(qa, orc.E5M2, orc.GRAN_TENSOR, sa),
                     orc.operand(qb, orc.E4M3, orc.GRAN_TENSOR, sb))
    yr, yar = _numpy_ref(qa, sa, orc.GRAN_TENSOR, orc.E5M2, qb, sb, orc.GRAN_TENSOR, orc.E4M3, M, N, K)
    assert np.all(np.abs(y - yr) <= 1e-13 * yar)


def test_gemm_scaled_identity_is_exact():
    # B = c * I on the first 128x128 block (c a power of two): y = deq(x) * c exactly
    M, K, N = 40, 256, 128
    x = inputs.activations(M, K, seed=9)
    qa, sa = orc.quantize_1x128(x, orc.E4M3, orc.SCALE_FP32)
    qb = np.zeros((N, K), np.uint8)
    qb[np.arange(128), np.arange(128)] = 0x38                     # 1.0 in E4M3
    sb = np.float32([[0.25, 1.0]])
    y, _ = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa),
                    orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb))
    deqx = _deq_codes(qa, orc.E4M3)[:, :128] * sa[0][:, None].astype(np.float64)
    assert np.array_equal(y, deqx * 0.25)


def test_gemm_integer_products_exact():
    rng = np.random.default_rng(1)
    M, N, K = 16, 24, 128
    # codes of small integers (E4M3: 1..8 exactly representable)
    ints = np.array([1, 2, 3, 4, 5, 6, 7, 8], dtype=np.float32)
    A = rng.choice(ints, size=(M, K)) * rng.choice([-1, 1], size=(M, K))
    B = rng.choice(ints, size=(N, K))
    qa = orc.encode_array(A.astype(np.float32), orc.E4M3)
    qb = orc.encode_array(B.astype(np.float32), orc.E4M3)
    one = np.float32([1.0])
    y, _ = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_TENSOR, one),
                    orc.operand(qb, orc.E4M3, orc.GRAN_TENSOR, one))
    assert np.array_equal(y, (A.astype(np.int64) @ B.astype(np.int64).T).astype(np.float64))


def test_grouped_gemm_vs_per_group_numpy():
    G, N, K = 5, 256, 256
    loads = np.array([3, 0, 130, 1, 60])                          # includes an empty group
    off = np.zeros(G + 1, np.int32)
    off[1:] = np.cumsum(loads)
    T = int(off[-1])
    x = inputs.gaussian((T + 7, K), 1.0, seed=12)                 # 7 rows beyond the last group
    w = inputs.gaussian((G * N, K), 0.02, seed=13)
    qa, sa = orc.quantize_1x128(x)
    qw, sw = [], []
    for g in range(G):
        q, s = orc.quantize_128x128(w[g * N:(g + 1) * N])
        qw.append(q)
        sw.append(s)
    qw, sw = np.concatenate(qw), np.stack(sw)
    A = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B = orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw)
    rows = np.array([0, 2, 3, 100, 132, 133, 134, 193, T, T + 6])
    y, ya = orc.grouped_gemm(off, T + 7, N, K, A, B, rows=rows)
    deqA = _deq_codes(qa, orc.E4M3) * _expand(sa, orc.GRAN_1x128, T + 7, K)
    for i, r in enumerate(rows):
        g = np.searchsorted(off, r, side="right") - 1
        if r >= T:
            assert np.all(np.isnan(y[i]))
            continue
        Bg = _deq_codes(qw[g * N:(g + 1) * N], orc.E4M3) * _expand(sw[g], orc.GRAN_128x128, N, K)
        ref = deqA[r] @ Bg.T
        assert np.all(np.abs(y[i] - ref) <= 1e-13 * ya[i])


def test_acceptance_rules():
    y_ref = np.array([1.0, -2.5, 1e-3, 0.0, 1000.0])
    yabs = np.array([10.0, 3.0, 1.0, 0.0, 2000.0])
    ok = y_ref + 0.9e-5 * yabs
    assert not orc.check_f32(ok.astype(np.float32), y_ref, yabs).any()
    bad = y_ref + 2e-5 * yabs
    assert orc.check_f32(bad, y_ref, yabs)[[0, 1, 2, 4]].all()
    # bf16: exact rounding and one step away pass, three steps fail
    b = orc._bf16_round(y_ref)
    assert not orc.check_bf16(b, y_ref, np.zeros(5)).any()
    assert not orc.check_bf16(b + 1, np.abs(y_ref), np.zeros(5))[[0, 2, 4]].any()
    assert orc.check_bf16(b + 3, np.abs(y_ref), np.zeros(5))[[0, 2, 4]].all()
