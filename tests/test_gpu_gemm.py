"""Parity of the tcgen05 block-scaled GEMM with the oracle.

Inputs are quantized by the ORACLE and uploaded, so the GEMM is checked on
its own.  fp32 output: |y - y_ref| <= 1e-5 * sum_k |terms| per element;
bf16 output: within one bf16 step of the rounding of a value inside that
bound (see oracle.check_bf16)."""
import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import dev, host, stratified

pytestmark = pytest.mark.gpu
REL = 1e-5


def _quant(bits, gran, fmt, mode):
    if gran == orc.GRAN_1x128:
        return orc.quantize_1x128(bits, fmt, mode)
    if gran == orc.GRAN_128x128:
        return orc.quantize_128x128(bits, fmt, mode)
    amax = float(np.abs(inputs.bits_to_f32(bits)).max())
    s = orc.block_scale(amax, fmt, mode)
    q, _ = orc.quantize_tensor(bits, fmt, s)
    return q, np.float32([s])


def _check(y_dev, y_ref, yabs, out_dtype, rows=None, cols=None):
    y = host(y_dev)
    if rows is not None:
        y = y[np.ix_(rows, cols)]
    if out_dtype == fp8.OUT_F32:
        bad = orc.check_f32(y, y_ref, yabs, REL)
    else:
        bad = orc.check_bf16(y.view(np.uint16), y_ref, yabs, REL)
    n_bad = int(bad.sum())
    if n_bad:
        i = np.argwhere(bad)[0]
        yv = y[tuple(i)]
        raise AssertionError(f"{n_bad}/{bad.size} outside tolerance; first {tuple(i)}: "
                             f"got {yv} ref {y_ref[tuple(i)]} abs {yabs[tuple(i)]}")


def _case(M, N, K, a_gran, b_gran, fa=orc.E4M3, fb=orc.E4M3, mode=orc.SCALE_FP32,
          a_t=False, b_t=False, seed=0):
    a = inputs.activations(M, K, seed=seed)
    b = inputs.gaussian((N, K), 0.02, seed=seed + 1)
    qa, sa = _quant(a, a_gran, fa, mode)
    qb, sb = _quant(b, b_gran, fb, mode)
    # storage of transposed operands: the matrix [K][rows], scale tables in
    # the stored orientation (a 128x128 table transposes with the matrix)
    sqa, ssa = (qa.T.copy(), sa.T.copy() if a_gran == orc.GRAN_128x128 else sa) if a_t else (qa, sa)
    sqb, ssb = (qb.T.copy(), sb.T.copy() if b_gran == orc.GRAN_128x128 else sb) if b_t else (qb, sb)
    A_o = orc.operand(sqa, fa, a_gran, ssa, transposed=a_t)
    B_o = orc.operand(sqb, fb, b_gran, ssb, transposed=b_t)
    A_d = fp8.operand(dev(sqa), dev(ssa), fa, a_gran, a_t)
    B_d = fp8.operand(dev(sqb), dev(ssb), fb, b_gran, b_t)
    return A_o, B_o, A_d, B_d


@pytest.mark.parametrize("out", [fp8.OUT_F32, fp8.OUT_BF16])
def test_tiny_config(out):
    """256x256x512, X 1x128 / W 128x128 E4M3, fp32 scales, full output."""
    M, N, K = 256, 256, 512
    A_o, B_o, A_d, B_d = _case(M, N, K, orc.GRAN_1x128, orc.GRAN_128x128)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    y = fp8.fp8_block_gemm(A_d, B_d, M, N, K, out)
    _check(y, y_ref, yabs, out)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (127, 256, 256), (129, 384, 640),
                                   (300, 520, 512), (513, 1024, 384), (64, 8, 128)])
@pytest.mark.parametrize("mode", [orc.SCALE_FP32, orc.SCALE_POW2])
def test_ragged_shapes(M, N, K, mode):
    A_o, B_o, A_d, B_d = _case(M, N, K, orc.GRAN_1x128, orc.GRAN_128x128, mode=mode, seed=M)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    for out in (fp8.OUT_F32, fp8.OUT_BF16):
        _check(fp8.fp8_block_gemm(A_d, B_d, M, N, K, out, mode), y_ref, yabs, out)


@pytest.mark.parametrize("a_gran,b_gran", [(orc.GRAN_128x128, orc.GRAN_128x128),
                                           (orc.GRAN_TENSOR, orc.GRAN_128x128),
                                           (orc.GRAN_1x128, orc.GRAN_TENSOR),
                                           (orc.GRAN_TENSOR, orc.GRAN_TENSOR)])
@pytest.mark.parametrize("mode", [orc.SCALE_FP32, orc.SCALE_POW2])
def test_granularities(a_gran, b_gran, mode):
    """fp32 scales: promotion kernel; pow2 scales: block-scaled (MX) kernel."""
    M, N, K = 200, 512, 1024
    A_o, B_o, A_d, B_d = _case(M, N, K, a_gran, b_gran, mode=mode, seed=7)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    _check(fp8.fp8_block_gemm(A_d, B_d, M, N, K, fp8.OUT_F32, mode), y_ref, yabs, fp8.OUT_F32)


@pytest.mark.parametrize("fa,fb", [(orc.E5M2, orc.E4M3), (orc.E4M3, orc.E5M2), (orc.E5M2, orc.E5M2)])
@pytest.mark.parametrize("mode", [orc.SCALE_FP32, orc.SCALE_POW2])
def test_mixed_formats(fa, fb, mode):
    M, N, K = 256, 256, 768
    A_o, B_o, A_d, B_d = _case(M, N, K, orc.GRAN_1x128, orc.GRAN_128x128, fa=fa, fb=fb, mode=mode,
                               seed=11)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    _check(fp8.fp8_block_gemm(A_d, B_d, M, N, K, fp8.OUT_F32, mode), y_ref, yabs, fp8.OUT_F32)


@pytest.mark.parametrize("a_t,b_t,a_gran,b_gran", [
    (False, True, orc.GRAN_1x128, orc.GRAN_128x128),     # dgrad, blockwise
    (False, True, orc.GRAN_TENSOR, orc.GRAN_TENSOR),     # dgrad, per-tensor
    (True, True, orc.GRAN_TENSOR, orc.GRAN_TENSOR),      # wgrad, per-tensor
    (True, True, orc.GRAN_128x128, orc.GRAN_128x128),    # wgrad, 128x128
    (True, False, orc.GRAN_TENSOR, orc.GRAN_128x128),
])
def test_transposed_operands(a_t, b_t, a_gran, b_gran):
    M, N, K = 384, 512, 640
    A_o, B_o, A_d, B_d = _case(M, N, K, a_gran, b_gran, fa=orc.E5M2, a_t=a_t, b_t=b_t, seed=13)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    _check(fp8.fp8_block_gemm(A_d, B_d, M, N, K, fp8.OUT_F32), y_ref, yabs, fp8.OUT_F32)


def test_k_zero_writes_zeros():
    import torch
    A = fp8.operand(torch.zeros((4, 16), dtype=torch.uint8, device="cuda"),
                    torch.ones((1, 4), device="cuda"), gran=fp8.GRAN_1x128)
    B = fp8.operand(torch.zeros((8, 16), dtype=torch.uint8, device="cuda"),
                    torch.ones((1, 1), device="cuda"), gran=fp8.GRAN_128x128)
    y = torch.full((4, 8), 7.0, device="cuda")
    fp8.fp8_block_gemm(A, B, 4, 8, 0, fp8.OUT_F32, y=y)
    assert torch.count_nonzero(y).item() == 0


def test_grouped_small():
    G, N, K = 6, 384, 512
    loads = np.array([0, 300, 1, 0, 129, 40])
    off = np.zeros(G + 1, np.int32)
    off[1:] = np.cumsum(loads)
    T = int(off[-1])
    a_rows = T + 5
    x = inputs.activations(a_rows, K, seed=31)
    w = inputs.gaussian((G * N, K), 0.02, seed=32)
    qa, sa = orc.quantize_1x128(x)
    qw = np.empty((G * N, K), np.uint8)
    sw = np.empty((G, (N + 127) // 128, K // 128), np.float32)
    for g in range(G):
        qw[g * N:(g + 1) * N], sw[g] = orc.quantize_128x128(w[g * N:(g + 1) * N])
    A_o = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B_o = orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw)
    y_ref, yabs = orc.grouped_gemm(off, a_rows, N, K, A_o, B_o, rows=np.arange(T))
    import torch
    y = torch.full((a_rows, N), float("nan"), device="cuda")
    fp8.fp8_grouped_block_gemm(dev(off), fp8.operand(dev(qa), dev(sa)),
                               fp8.operand(dev(qw), dev(sw), gran=fp8.GRAN_128x128),
                               a_rows, N, K, fp8.OUT_F32, y=y)
    yh = host(y)
    bad = orc.check_f32(yh[:T], y_ref, yabs, REL)
    assert not bad.any(), int(bad.sum())
    assert np.all(np.isnan(yh[T:]))            # rows outside every group untouched


def test_back_to_back_calls_and_side_stream():
    import torch
    M, N, K = 300, 512, 512
    A_o, B_o, A_d, B_d = _case(M, N, K, orc.GRAN_1x128, orc.GRAN_128x128, seed=41)
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ys = [fp8.fp8_block_gemm(A_d, B_d, M, N, K, fp8.OUT_F32) for _ in range(3)]
    s.synchronize()
    for y in ys:
        _check(y, y_ref, yabs, fp8.OUT_F32)
    fp8.device_status()


def test_pow2_scale_extremes_mx():
    """Block-scaled (MX) path with scales spread over a wide exponent range,
    per-row and per-block (tiny and huge blocks side by side)."""
    M, N, K = 256, 512, 512
    rng = np.random.default_rng(21)
    a = inputs.bits_to_f32(inputs.activations(M, K, seed=21))
    a *= (2.0 ** rng.integers(-40, 40, size=(M, 1))).astype(np.float32)
    b = inputs.bits_to_f32(inputs.gaussian((N, K), 0.02, seed=22))
    b *= (2.0 ** rng.integers(-30, 30, size=(N // 128, 1))).repeat(128, axis=0).astype(np.float32)
    qa, sa = orc.quantize_1x128(inputs.bf16_bits(a), orc.E4M3, orc.SCALE_POW2)
    qb, sb = orc.quantize_128x128(inputs.bf16_bits(b), orc.E4M3, orc.SCALE_POW2)
    y_ref, yabs = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa),
                           orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb))
    y = fp8.fp8_block_gemm(fp8.operand(dev(qa), dev(sa)), fp8.operand(dev(qb), dev(sb), gran=fp8.GRAN_128x128),
                           M, N, K, fp8.OUT_F32, fp8.SCALE_POW2)
    _check(y, y_ref, yabs, fp8.OUT_F32)


# ------------------------------------------------------------ full sizes
LLAMA8B = [("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 28672, 4096), ("down", 4096, 14336)]


LLAMA2 = [("qkv", 12288, 4096), ("down", 4096, 11008)]


@pytest.mark.parametrize("name,N,K", LLAMA2)
def test_llama2_7b_pow2_linears_sampled(name, N, K):
    """Llama-2-7B-shaped linears (M=4096) with power-of-two scales: the
    block-scaled (MX) kernel at full size, sampled outputs."""
    M = 4096
    x = inputs.activations(M, K, seed=3000 + K)
    w = inputs.gaussian((N, K), 0.02, seed=4000 + N)
    qa, sa = orc.quantize_1x128(x, orc.E4M3, orc.SCALE_POW2)
    qb, sb = orc.quantize_128x128(w, orc.E4M3, orc.SCALE_POW2)
    rng = np.random.default_rng(N)
    rows, cols = stratified(M, 128, rng), stratified(N, 256, rng, extra=(N - 8,))
    y_ref, yabs = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa),
                           orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb), rows=rows, cols=cols)
    A_d = fp8.operand(dev(qa), dev(sa))
    B_d = fp8.operand(dev(qb), dev(sb), gran=fp8.GRAN_128x128)
    for out in (fp8.OUT_BF16, fp8.OUT_F32):
        _check(fp8.fp8_block_gemm(A_d, B_d, M, N, K, out, fp8.SCALE_POW2), y_ref, yabs, out, rows, cols)


@pytest.mark.parametrize("name,N,K", LLAMA8B)
def test_llama31_8b_linears_sampled(name, N, K):
    """Full Llama-3.1-8B-shaped fprop linears (M=8192, fp32 scales, bf16 out as
    the benchmark runs them), checked on one sampled row per 128-row block and
    one sampled column per 256-column block."""
    M = 8192
    x = inputs.activations(M, K, seed=1000 + K)
    w = inputs.gaussian((N, K), 0.02, seed=2000 + N)
    qa, sa = orc.quantize_1x128(x)
    qb, sb = orc.quantize_128x128(w)
    A_o = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B_o = orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb)
    rng = np.random.default_rng(N + K)
    rows = stratified(M, 128, rng)
    cols = stratified(N, 256, rng, extra=(N - 8,))
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o, rows=rows, cols=cols)
    A_d = fp8.operand(dev(qa), dev(sa))
    B_d = fp8.operand(dev(qb), dev(sb), gran=fp8.GRAN_128x128)
    for out in (fp8.OUT_BF16, fp8.OUT_F32):
        y = fp8.fp8_block_gemm(A_d, B_d, M, N, K, out)
        _check(y, y_ref, yabs, out, rows, cols)


# ------------------------------------- many tiles per CTA, many groups
@pytest.mark.parametrize("a_t,b_t,a_gran,b_gran,fa", [
    (False, True, orc.GRAN_1x128, orc.GRAN_128x128, orc.E4M3),   # dgrad, blockwise
    (False, True, orc.GRAN_TENSOR, orc.GRAN_TENSOR, orc.E5M2),   # dgrad, per-tensor (whole K in TMEM)
    (True, True, orc.GRAN_TENSOR, orc.GRAN_TENSOR, orc.E5M2),    # wgrad, per-tensor (whole K in TMEM)
    (True, True, orc.GRAN_128x128, orc.GRAN_128x128, orc.E4M3),  # wgrad, 128x128
    (True, False, orc.GRAN_TENSOR, orc.GRAN_128x128, orc.E5M2),
    (False, False, orc.GRAN_TENSOR, orc.GRAN_TENSOR, orc.E5M2),  # K-major, whole K in TMEM
])
def test_transposed_operands_many_tiles_per_cta(a_t, b_t, a_gran, b_gran, fa):
    """32 x 10 = 320 output tiles on 152 persistent CTAs: every CTA takes two or
    three tiles, so the TMEM buffers and every barrier phase are reused across
    tiles; every tile is sampled (two rows per 128-row block, two columns per
    256-column block)."""
    M, N, K = 4096, 2560, 512
    A_o, B_o, A_d, B_d = _case(M, N, K, a_gran, b_gran, fa=fa, a_t=a_t, b_t=b_t, seed=17)
    rng = np.random.default_rng(M + N)
    rows = np.unique(np.concatenate([stratified(M, 128, rng), stratified(M, 128, rng)]))
    cols = np.unique(np.concatenate([stratified(N, 256, rng), stratified(N, 256, rng)]))
    y_ref, yabs = orc.gemm(M, N, K, A_o, B_o, rows=rows, cols=cols)
    for out in (fp8.OUT_F32, fp8.OUT_BF16):
        _check(fp8.fp8_block_gemm(A_d, B_d, M, N, K, out), y_ref, yabs, out, rows, cols)
    fp8.device_status()


def _grouped_operands(loads, N, K, seed, extra_rows=0):
    G = loads.size
    off = np.zeros(G + 1, np.int32)
    off[1:] = np.cumsum(loads)
    T = int(off[-1])
    a_rows = T + extra_rows
    x = inputs.activations(a_rows, K, seed=seed)
    w = inputs.gaussian((G * N, K), 0.02, seed=seed + 1)
    qa, sa = orc.quantize_1x128(x)
    qw, sw = orc.quantize_128x128(w)
    sw = sw.reshape(G, (N + 127) // 128, K // 128)
    return off, T, a_rows, qa, sa, qw, sw


def test_grouped_more_than_32_groups():
    """40 groups (the device prefix of m-slots runs over two 32-group chunks):
    empty, 1-row, exactly-128-row and multi-slot groups; 5 rows past the last
    group stay untouched."""
    import torch
    rng = np.random.default_rng(41)
    loads = rng.integers(0, 300, 40)
    loads[[0, 7, 33]] = 0
    loads[[3, 35]] = 1
    loads[[12, 39]] = 128
    N, K = 384, 256
    off, T, a_rows, qa, sa, qw, sw = _grouped_operands(loads, N, K, seed=43, extra_rows=5)
    A_o = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B_o = orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw)
    y_ref, yabs = orc.grouped_gemm(off, a_rows, N, K, A_o, B_o, rows=np.arange(T))
    y = torch.full((a_rows, N), float("nan"), device="cuda")
    fp8.fp8_grouped_block_gemm(dev(off), fp8.operand(dev(qa), dev(sa)),
                               fp8.operand(dev(qw), dev(sw), gran=fp8.GRAN_128x128),
                               a_rows, N, K, fp8.OUT_F32, y=y)
    fp8.device_status()
    yh = host(y)
    _check(y[:T], y_ref, yabs, fp8.OUT_F32)
    assert np.all(np.isnan(yh[T:]))


def test_grouped_maximum_group_count():
    """1024 groups, the most one call takes (empty, 1-row and multi-slot groups;
    the device prefix of m-slots spans 32 chunks), sampled rows of every group
    and all columns; rows past the last group stay untouched."""
    import torch
    from helpers import par_grouped_gemm
    rng = np.random.default_rng(51)
    loads = rng.integers(0, 200, 1024)
    loads[rng.choice(1024, 100, replace=False)] = 0
    loads[rng.choice(1024, 50, replace=False)] = 1
    N, K = 256, 256
    off, T, a_rows, qa, sa, qw, sw = _grouped_operands(loads, N, K, seed=53, extra_rows=3)
    rows = np.unique(np.concatenate([off[:-1][loads > 0], off[1:][loads > 0] - 1,
                                     rng.integers(0, T, 2000)]))
    A_o = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B_o = orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw)
    y_ref, yabs = par_grouped_gemm(orc, off, a_rows, N, K, A_o, B_o, rows, np.arange(N))
    y = torch.full((a_rows, N), float("nan"), device="cuda")
    fp8.fp8_grouped_block_gemm(dev(off), fp8.operand(dev(qa), dev(sa)),
                               fp8.operand(dev(qw), dev(sw), gran=fp8.GRAN_128x128),
                               a_rows, N, K, fp8.OUT_F32, y=y)
    fp8.device_status()
    yh = host(y)
    _check(y, y_ref, yabs, fp8.OUT_F32, rows, np.arange(N))
    assert np.all(np.isnan(yh[T:]))


def test_grouped_all_groups_empty_writes_nothing():
    import torch
    loads = np.zeros(5, np.int64)
    N, K = 256, 128
    off, T, a_rows, qa, sa, qw, sw = _grouped_operands(loads, N, K, seed=57, extra_rows=7)
    y = torch.full((a_rows, N), float("nan"), device="cuda")
    fp8.fp8_grouped_block_gemm(dev(off), fp8.operand(dev(qa), dev(sa)),
                               fp8.operand(dev(qw), dev(sw), gran=fp8.GRAN_128x128),
                               a_rows, N, K, fp8.OUT_F32, y=y)
    fp8.device_status()
    assert T == 0 and np.all(np.isnan(host(y)))


def test_grouped_decreasing_offsets_are_reported_and_nothing_is_written():
    """A decreasing offset table would give overlapping groups (two tiles
    writing the same rows).  The kernel writes nothing and the device status
    reports an invalid argument; the next product runs normally."""
    import torch
    loads = np.array([200, 100, 150])
    N, K = 256, 256
    off, T, a_rows, qa, sa, qw, sw = _grouped_operands(loads, N, K, seed=47)
    A_d = fp8.operand(dev(qa), dev(sa))
    B_d = fp8.operand(dev(qw), dev(sw), gran=fp8.GRAN_128x128)
    bad_off = np.array([0, 200, 120, 450], np.int32)      # group 1 ends before it starts
    y = torch.full((a_rows, N), float("nan"), device="cuda")
    fp8.fp8_grouped_block_gemm(dev(bad_off), A_d, B_d, a_rows, N, K, fp8.OUT_F32, y=y)
    with pytest.raises(fp8.Fp8bsError) as e:
        fp8.device_status()
    assert e.value.code == -1
    assert np.all(np.isnan(host(y)))
    fp8.device_status()                                   # the record was cleared
    y_ref, yabs = orc.grouped_gemm(off, a_rows, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa),
                                   orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw), rows=np.arange(T))
    fp8.fp8_grouped_block_gemm(dev(off), A_d, B_d, a_rows, N, K, fp8.OUT_F32, y=y)
    fp8.device_status()
    _check(y[:T], y_ref, yabs, fp8.OUT_F32)


def test_pow2_mode_with_per_tensor_scales_that_are_not_powers_of_two():
    """Under POW2 the block scales are powers of two, but a per-tensor scale
    (delayed scaling: amax_history / fmax) in general is not; such products
    must still give the exact sum."""
    M, N, K = 256, 512, 512
    a = inputs.activations(M, K, seed=53)
    b = inputs.gaussian((N, K), 0.02, seed=54)
    amax = float(np.abs(inputs.bits_to_f32(a)).max())
    s_t = np.float32([amax / 448.0 * 1.37])               # not a power of two
    qa, _ = orc.quantize_tensor(a, orc.E4M3, float(s_t[0]))
    qb, sb = orc.quantize_128x128(b, orc.E4M3, orc.SCALE_POW2)
    y_ref, yabs = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_TENSOR, s_t),
                           orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb))
    y = fp8.fp8_block_gemm(fp8.operand(dev(qa), dev(s_t), gran=fp8.GRAN_TENSOR),
                           fp8.operand(dev(qb), dev(sb), gran=fp8.GRAN_128x128), M, N, K, fp8.OUT_F32,
                           fp8.SCALE_POW2)
    _check(y, y_ref, yabs, fp8.OUT_F32)


def _block_varying(x_bits, K, seed):
    """Activations whose magnitude changes by up to 2^4 from one 128-column
    block to the next (and between rows), so that a scale applied to the
    wrong K block or row moves the result far outside the tolerance."""
    x = inputs.bits_to_f32(x_bits).astype(np.float64)
    rng = np.random.default_rng(seed)
    blk = 2.0 ** rng.integers(-2, 3, size=(x.shape[0] // 64 + 1, K // 128))
    f = np.repeat(np.repeat(blk, 64, axis=0)[:x.shape[0]], 128, axis=1)
    return inputs.bf16_bits((x * f).astype(np.float32))


def test_repeated_grouped_runs_are_identical_and_match_the_oracle():
    """Many tiles per CTA with a short K (the scale ring and the two TMEM
    buffers wrap many times per tile sequence) on 64 experts with ragged
    group starts: eight launches give bit-identical outputs, and every row of
    the first is checked against the oracle on sampled columns."""
    import torch
    from helpers import par_grouped_gemm
    rng = np.random.default_rng(77)
    G, N, K = 64, 1024, 768
    loads = rng.integers(1, 1500, G)
    off = np.concatenate([[0], np.cumsum(loads)]).astype(np.int32)
    T = int(off[-1])
    x = _block_varying(inputs.activations(T, K, seed=78), K, seed=79)
    w = inputs.gaussian((G * N, K), 0.02, seed=80)
    qa, sa = orc.quantize_1x128(x)
    qw, sw = orc.quantize_128x128(w)
    sw = sw.reshape(G, N // 128, K // 128)
    A_o = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B_o = orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw)
    A_d = fp8.operand(dev(qa), dev(sa))
    B_d = fp8.operand(dev(qw), dev(sw), gran=fp8.GRAN_128x128)
    offd = dev(off)
    ys = [fp8.fp8_grouped_block_gemm(offd, A_d, B_d, T, N, K, fp8.OUT_BF16) for _ in range(8)]
    fp8.device_status()
    for i in range(1, 8):
        assert torch.equal(ys[i], ys[0]), f"launch {i} differs from launch 0"
    cols = stratified(N, 128, rng, extra=(N - 1,))
    rows = np.arange(T)
    y_ref, yabs = par_grouped_gemm(orc, off, T, N, K, A_o, B_o, rows, cols)
    _check(ys[0], y_ref, yabs, fp8.OUT_BF16, rows=rows, cols=cols)


@pytest.mark.parametrize("M", [4096, 4093])
def test_repeated_dense_runs_are_identical_and_match_the_oracle(M):
    """A dense product with several tiles per CTA and 48 K blocks, with the
    1x128 scale table aligned (copied by the producer) and, for M = 4093,
    not (staged by the scale warp's own loads): eight launches give
    bit-identical outputs; sampled rows and columns match the oracle."""
    import torch
    from helpers import par_gemm
    rng = np.random.default_rng(M)
    N, K = 2048, 6144
    x = _block_varying(inputs.activations(M, K, seed=81), K, seed=82)
    w = inputs.gaussian((N, K), 0.02, seed=83)
    qa, sa = orc.quantize_1x128(x)
    qw, sw = orc.quantize_128x128(w)
    A_o = orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa)
    B_o = orc.operand(qw, orc.E4M3, orc.GRAN_128x128, sw)
    A_d = fp8.operand(dev(qa), dev(sa))
    B_d = fp8.operand(dev(qw), dev(sw), gran=fp8.GRAN_128x128)
    ys = [fp8.fp8_block_gemm(A_d, B_d, M, N, K, fp8.OUT_BF16) for _ in range(8)]
    fp8.device_status()
    for i in range(1, 8):
        assert torch.equal(ys[i], ys[0]), f"launch {i} differs from launch 0"
    rows = stratified(M, 128, rng, extra=(M - 1,))
    cols = stratified(N, 128, rng, extra=(N - 1,))
    y_ref, yabs = par_gemm(orc, M, N, K, A_o, B_o, rows, cols)
    _check(ys[0], y_ref, yabs, fp8.OUT_BF16, rows=rows, cols=cols)
