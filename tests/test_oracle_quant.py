"""Pins of the oracle's block quantizers and delayed-scaling state machine.

Independent checks, none of which re-types the oracle's C code:
- power-of-two scales worked by hand (golden file) and a brute-force search
  over exponents done in Python integers;
- tile partitioning checked with numpy reshapes and an encoder that is a
  nearest-entry search over PyTorch's float8 decode table;
- invariants: the block maximum lands on +-fmax (fp32 scales), never
  saturates (pow2 scales), dequantization error within half a grid step;
- the delayed-scaling closed form: with a history that never wraps the scale
  in use at step t is max(amax_0..amax_{t-1}) / fmax.
"""
import os

import numpy as np
import pytest
import torch

import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMAX = {orc.E4M3: 448.0, orc.E5M2: 57344.0}
TORCH_T = {orc.E4M3: torch.float8_e4m3fn, orc.E5M2: torch.float8_e5m2}


def _table(fmt):
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(TORCH_T[fmt]).to(torch.float64).numpy()


def _nearest_code(v: np.ndarray, fmt: int) -> np.ndarray:
    """Nearest-entry search in torch's decode table, ties to even, saturating."""
    t = _table(fmt)
    maxcode = 0x7E if fmt == orc.E4M3 else 0x7B
    mags = t[: maxcode + 1]
    a = np.abs(v.astype(np.float64))
    hi = np.clip(np.searchsorted(mags, a), 0, maxcode)
    lo = np.clip(np.searchsorted(mags, a) - 1, 0, maxcode)
    dlo, dhi = a - mags[lo], mags[hi] - a
    pick = np.where(dlo < dhi, lo, hi)
    pick = np.where((dlo == dhi) & (lo != hi), np.where(lo % 2 == 0, lo, hi), pick)
    pick = np.where(a >= mags[-1], maxcode, pick)
    return (pick | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)


def _expected_block_quant(xf: np.ndarray, amax: np.ndarray, fmt: int, mode: int):
    """Expected (q, s) for elements xf with their block amax broadcast."""
    if mode == orc.SCALE_FP32:
        s = np.where(amax > 0, np.maximum(amax / np.float32(FMAX[fmt]), np.float32(2.0 ** -126)),
                     np.float32(1.0)).astype(np.float32)
    else:
        uniq, inv = np.unique(amax.ravel(), return_inverse=True)
        su = np.array([_pow2_bruteforce(float(a), fmt) for a in uniq], dtype=np.float32)
        s = su[inv].reshape(amax.shape)
    r = (np.float32(1.0) / s).astype(np.float32)
    v = (xf * r).astype(np.float32)
    return _nearest_code(v, fmt), s


def _pow2_bruteforce(amax: float, fmt: int) -> float:
    if not amax > 0:
        return 1.0
    from fractions import Fraction
    a = Fraction(amax)
    for e in range(-126, 128):
        if a <= Fraction(int(FMAX[fmt])) * (Fraction(2) ** e):
            return 2.0 ** e
    return 2.0 ** 127


def test_pow2_golden_examples():
    n = 0
    with open(os.path.join(GOLDEN, "pow2_scale_examples.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            fmt, amax, want = line.split()
            fmt = orc.E4M3 if fmt == "e4m3" else orc.E5M2
            assert orc.block_scale(float(amax), fmt, orc.SCALE_POW2) == float(want), line
            n += 1
    assert n >= 9


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_pow2_rule_bruteforce_and_invariant(fmt):
    rng = np.random.default_rng(3)
    amaxes = np.concatenate([
        (10.0 ** rng.uniform(-38, 38, 3000)).astype(np.float32),
        inputs.bits_to_f32(rng.integers(0x0001, 0x7F80, 3000).astype(np.uint16)),  # all bf16 magnitudes
        np.float32([2.0 ** -149, 2.0 ** -126, 448.0, 57344.0, 1.75, 3.5]),
    ])
    for a in amaxes:
        s = orc.block_scale(float(a), fmt, orc.SCALE_POW2)
        assert s == _pow2_bruteforce(float(a), fmt)
        e = int(np.log2(s))
        if -126 < e:
            assert FMAX[fmt] / 2 < a / s <= FMAX[fmt]


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_fp32_scale_examples(fmt):
    assert orc.block_scale(0.0, fmt, orc.SCALE_FP32) == 1.0
    assert orc.block_scale(FMAX[fmt], fmt, orc.SCALE_FP32) == 1.0
    assert orc.block_scale(2 * FMAX[fmt], fmt, orc.SCALE_FP32) == 2.0
    assert orc.block_scale(1e-40, fmt, orc.SCALE_FP32) == 2.0 ** -126     # floor
    # correctly rounded quotient: 1/448 = 0.00223214285714...; nearest fp32
    want = float(np.float32(np.float64(1.0) / FMAX[fmt]))
    assert orc.block_scale(1.0, fmt, orc.SCALE_FP32) == want


@pytest.mark.parametrize("mode", [orc.SCALE_FP32, orc.SCALE_POW2])
@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_quantize_1x128_tiles(fmt, mode):
    M, K = 37, 384
    x = inputs.activations(M, K, seed=11)
    x[3, 128:256] = 0                              # an all-zero tile
    x[5, 0] = 0x8000                               # a -0
    q, s = orc.quantize_1x128(x, fmt, mode)
    xf = inputs.bits_to_f32(x)
    amax = np.abs(xf).reshape(M, K // 128, 128).max(axis=2)           # [M, K/128]
    want_q, want_s = _expected_block_quant(xf, np.repeat(amax, 128, axis=1), fmt, mode)
    assert np.array_equal(q, want_q)
    assert np.array_equal(s, want_s[:, ::128].T)                      # layout [K/128][M]
    assert s.shape == (K // 128, M)
    assert s[1, 3] == 1.0 and np.all(q[3, 128:256] == 0)
    assert q[5, 0] == 0x80
    t = _table(fmt)
    deq = t[q] * np.repeat(s.T, 128, axis=1)
    # the maximum of each block is never saturated away: fp32 scales put it
    # on +-fmax exactly, pow2 scales within (fmax/2, fmax]
    blk_max = np.abs(deq).reshape(M, K // 128, 128).max(axis=2)
    nz = amax > 0
    if mode == orc.SCALE_FP32:
        assert np.all(np.abs(t[q]).reshape(M, K // 128, 128).max(axis=2)[nz] == FMAX[fmt])
    # dequantization error: at most half a grid step of the format (relative
    # 2^-4 for E4M3, 2^-3 for E5M2 in the normal range) plus subnormal spacing
    rel = 2.0 ** -4 if fmt == orc.E4M3 else 2.0 ** -3
    sub = (2.0 ** -10 if fmt == orc.E4M3 else 2.0 ** -17) * np.repeat(s.T, 128, axis=1)
    assert np.all(np.abs(deq - xf) <= rel * np.abs(xf) + sub * 1.0001)
    assert np.all(blk_max <= amax * (1 + rel) + 1e-30)


@pytest.mark.parametrize("mode", [orc.SCALE_FP32, orc.SCALE_POW2])
def test_quantize_128x128_tiles(mode):
    N, K = 300, 256                                # ragged last row-tile (44 rows)
    w = inputs.gaussian((N, K), 0.02, seed=5)
    q, s = orc.quantize_128x128(w, orc.E4M3, mode)
    assert s.shape == (3, 2)
    wf = inputs.bits_to_f32(w)
    pad = np.zeros((384, K), dtype=np.float32)
    pad[:N] = np.abs(wf)
    amax = pad.reshape(3, 128, 2, 128).max(axis=(1, 3))              # [3, 2]
    amax_el = np.repeat(np.repeat(amax, 128, axis=0), 128, axis=1)[:N]
    want_q, want_s = _expected_block_quant(wf, amax_el, orc.E4M3, mode)
    assert np.array_equal(q, want_q)
    assert np.array_equal(s, want_s[::128, ::128])


def test_quantize_is_tile_local():
    # changing one tile changes only that tile's codes and scale
    M, K = 8, 512
    x = inputs.activations(M, K, seed=2)
    q0, s0 = orc.quantize_1x128(x)
    x2 = x.copy()
    x2[4, 256:384] = inputs.bf16_bits(np.full(128, 1000.0, np.float32))
    q1, s1 = orc.quantize_1x128(x2)
    diff = np.argwhere(q0 != q1)
    assert np.all(diff[:, 0] == 4) and np.all((diff[:, 1] >= 256) & (diff[:, 1] < 384))
    sd = np.argwhere(s0 != s1)
    assert sd.tolist() == [[2, 4]]


def test_quantize_tensor_and_amax():
    x = inputs.student_t((64, 256), 3.0, 1e-3, seed=100)
    xf = inputs.bits_to_f32(x)
    for scale in (1.0, 3.7e-7, 2.0 ** -20):
        q, amax = orc.quantize_tensor(x, orc.E5M2, scale)
        assert amax == np.abs(xf).max()
        r = np.float32(1.0) / np.float32(scale)
        assert np.array_equal(q.ravel(), _nearest_code((xf.ravel() * r).astype(np.float32), orc.E5M2))


def test_delayed_closed_form_no_wrap():
    # history length 1024, 16 steps: scale_t = max(amax_0..amax_{t-1}) / fmax,
    # step 0 uses scale 1 (introl: scales from earlier iterations' maxima).
    st = orc.DelayedState(1024, orc.E5M2, margin=0)
    amaxes = []
    for t in range(16):
        x = inputs.student_t((32, 128), 3.0, 1e-3 * (1 + (t % 5)), seed=100 + t)
        want_scale = 1.0 if t == 0 else float(np.float32(max(amaxes)) / np.float32(57344.0))
        assert float(st.scale[0]) == want_scale
        q, amax = st.step(x)
        amaxes.append(amax)
    assert int(st.head[0]) == 16


def test_delayed_wraps_and_margin():
    st = orc.DelayedState(4, orc.E4M3, margin=2)
    seq = [8.0, 2.0, 1.0, 0.5, 0.25, 0.125]
    got = [st.update(a) for a in seq]
    # window of the last 4 amaxes, times 2^margin, over 448
    want = []
    for i in range(len(seq)):
        m = max(seq[max(0, i - 3): i + 1])
        want.append(float(np.float32(np.float32(m) / np.float32(448.0)) * np.float32(4.0)))
    assert got == want
    assert int(st.head[0]) == len(seq) % 4


def test_delayed_zero_history_keeps_scale():
    st = orc.DelayedState(4, orc.E4M3)
    assert st.update(0.0) == 1.0
    st.update(448.0)
    assert float(st.scale[0]) == 1.0
    for _ in range(3):
        st.update(0.0)
    assert float(st.scale[0]) == 1.0          # 448 still inside the window
    st.update(0.0)                             # window all zero -> scale kept
    assert float(st.scale[0]) == 1.0


def test_delayed_save_restore_bit_identical():
    xs = [inputs.student_t((16, 128), 3.0, 1e-3, seed=200 + t) for t in range(16)]
    a = orc.DelayedState(8, orc.E5M2)
    qa = [a.step(x)[0] for x in xs]
    b = orc.DelayedState(8, orc.E5M2)
    qb = [b.step(x)[0] for x in xs[:8]]
    saved = (b.history.copy(), b.head.copy(), b.scale.copy())
    c = orc.DelayedState(8, orc.E5M2)
    c.history[:], c.head[:], c.scale[:] = saved
    qb += [c.step(x)[0] for x in xs[8:]]
    assert all(np.array_equal(u, v) for u, v in zip(qa, qb))
    assert np.array_equal(a.history, c.history) and a.scale[0] == c.scale[0]
