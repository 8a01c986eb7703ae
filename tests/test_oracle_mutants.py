"""Planted mistakes: each test compiles a copy of the oracle with one plausible
bug (a dropped rule, a wrong sign, index or rounding direction) and checks
that an independent pin -- the same kinds of references the oracle pins use
(PyTorch's float8 decode, a brute-force nearest-code search, numpy tile
reductions, numpy fp64 matmul, closed forms) -- rejects it.  The mistakes
live only in these compiled copies, on the CPU."""
import numpy as np
import pytest
import torch

import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs


def _nearest_code(v, fmt):
    t = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn if fmt == orc.E4M3 else torch.float8_e5m2).to(torch.float64).numpy()
    maxcode = 0x7E if fmt == orc.E4M3 else 0x7B
    mags = t[: maxcode + 1]
    a = np.abs(np.asarray(v, np.float64))
    hi = np.clip(np.searchsorted(mags, a), 0, maxcode)
    lo = np.clip(np.searchsorted(mags, a) - 1, 0, maxcode)
    dlo, dhi = a - mags[lo], mags[hi] - a
    pick = np.where(dlo < dhi, lo, hi)
    pick = np.where((dlo == dhi) & (lo != hi), np.where(lo % 2 == 0, lo, hi), pick)
    pick = np.where(a >= mags[-1], maxcode, pick)
    return (pick | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)


def _encoder_pin():
    """Midpoints, saturation, signed zero and a random sweep vs brute force."""
    for fmt in (orc.E4M3, orc.E5M2):
        t = orc.decode_table(fmt)
        maxcode = 0x7E if fmt == orc.E4M3 else 0x7B
        mids = np.float32([(t[c] + t[c + 1]) / 2 for c in range(maxcode)])
        rng = np.random.default_rng(0)
        v = np.concatenate([mids, -mids, np.float32([470.0, 1e30, -0.0, -1e-30, 61440.0]),
                            (rng.standard_normal(20000) * 10.0 ** rng.uniform(-6, 5, 20000)).astype(np.float32)])
        if not np.array_equal(orc.encode_array(v, fmt), _nearest_code(v, fmt)):
            return False
    return True


def _decode_pin():
    for fmt, tt in ((orc.E4M3, torch.float8_e4m3fn), (orc.E5M2, torch.float8_e5m2)):
        ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(tt).to(torch.float64).numpy()
        got = orc.decode_table(fmt)
        m = ~np.isnan(ref)
        if not (np.array_equal(np.isnan(ref), np.isnan(got)) and np.array_equal(ref[m], got[m])):
            return False
    return True


def _tile_pin():
    """1x128 and 128x128 tiles vs numpy reductions + the brute-force encoder."""
    M, K = 20, 384
    x = inputs.activations(M, K, seed=1)
    q, s = orc.quantize_1x128(x)
    xf = inputs.bits_to_f32(x)
    amax = np.abs(xf).reshape(M, K // 128, 128).max(axis=2)
    want_s = (amax / np.float32(448.0)).astype(np.float32)
    r = (np.float32(1.0) / np.repeat(want_s, 128, axis=1)).astype(np.float32)
    if s.shape != (K // 128, M) or not np.array_equal(s, want_s.T):
        return False
    if not np.array_equal(q, _nearest_code((xf * r).astype(np.float32), orc.E4M3)):
        return False
    w = inputs.gaussian((130, 256), 0.02, seed=2)
    q2, s2 = orc.quantize_128x128(w)
    pad = np.zeros((256, 256), np.float32)
    pad[:130] = np.abs(inputs.bits_to_f32(w))
    am2 = pad.reshape(2, 128, 2, 128).max(axis=(1, 3))
    return np.array_equal(s2, (am2 / np.float32(448.0)).astype(np.float32))


def _pow2_pin():
    examples = [(448.0, 1.0), (450.0, 2.0), (1.0, 2.0 ** -8), (1.75, 2.0 ** -8), (0.875, 2.0 ** -9)]
    return all(orc.block_scale(a, orc.E4M3, orc.SCALE_POW2) == s for a, s in examples)


def _gemm_pin():
    M, N, K = 24, 136, 256
    qa, sa = orc.quantize_1x128(inputs.activations(M, K, seed=3))
    qb, sb = orc.quantize_128x128(inputs.gaussian((N, K), 0.02, seed=4))
    y, ya = orc.gemm(M, N, K, orc.operand(qa, orc.E4M3, orc.GRAN_1x128, sa),
                     orc.operand(qb, orc.E4M3, orc.GRAN_128x128, sb))
    dec = lambda q: torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    A = dec(qa) * np.repeat(sa.T.astype(np.float64), 128, axis=1)
    B = dec(qb) * np.repeat(np.repeat(sb.astype(np.float64), 128, axis=0), 128, axis=1)[:N]
    return bool(np.all(np.abs(y - A @ B.T) <= 1e-12 * (np.abs(A) @ np.abs(B).T)))


def _delayed_pin():
    st = orc.DelayedState(4, orc.E4M3, margin=0)
    seq = [8.0, 2.0, 1.0, 0.5, 0.25, 0.125]
    got = [st.update(a) for a in seq]
    want = [float(np.float32(max(seq[max(0, i - 3): i + 1])) / np.float32(448.0)) for i in range(6)]
    return got == want


def _f32_tile_pin():
    """1x128 rule on fp32 input vs numpy reductions + the brute-force encoder."""
    rng = np.random.default_rng(9)
    y = (rng.standard_normal((6, 256)) * 5).astype(np.float32)
    y[0, 127], y[1, 255], y[2, 128] = 100.0, -100.0, 90.0   # block maxima at the block edges
    q, s = orc.quantize_1x128_f32(y)
    amax = np.abs(y).reshape(6, 2, 128).max(axis=2)
    want = (amax / np.float32(448.0)).astype(np.float32)
    r = (np.float32(1.0) / np.repeat(want, 128, axis=1)).astype(np.float32)
    return bool(np.array_equal(s, want.T) and
                np.array_equal(q, _nearest_code((y * r).astype(np.float32), orc.E4M3)))


PINS = [_encoder_pin, _decode_pin, _tile_pin, _pow2_pin, _gemm_pin, _delayed_pin, _f32_tile_pin]

MUTANTS = {
    "ties_away_from_zero": ("if (rem > half || (rem == half && (n & 1))) n += 1;",
                            "if (rem >= half) n += 1;"),
    "no_saturation_at_fmax": ("if (mag > f.maxcode) mag = f.maxcode;",
                              "if (mag > f.maxcode + 1) mag = f.maxcode;"),
    "signed_zero_dropped": ("if (a < 0x00800000u) return sign;", "if (a < 0x00800000u) return 0;"),
    "e4m3_subnormal_exponent": ("return sign * ldexp((double)m, -9);", "return sign * ldexp((double)m, -8);"),
    "scale_divides_by_fmax_minus_1": ("float s = amax / (float)f.fmax;",
                                      "float s = amax / ((float)f.fmax - 1.0f);"),
    "pow2_rounds_strictly": ("if ((double)amax <= ldexp(f.fmax, e)) break;",
                             "if ((double)amax < ldexp(f.fmax, e)) break;"),
    "scale_table_transposed": ("scales[kb * rows + r] = s;", "scales[r * nkb + kb] = s;"),
    "gemm_first_term_sign": ("acc += p;", "acc += (k == 0 ? -p : p);"),
    "history_head_stuck": ("*head = (*head + 1) % L;", "*head = (*head) % L;"),
    "amax_without_abs": ("float a = fabsf(fp8o_bf16_to_f32(x[r * ldx + c]));",
                         "float a = fp8o_bf16_to_f32(x[r * ldx + c]);"),
    "f32_amax_without_abs": ("float a = fabsf(y[r * ldy + c]);", "float a = y[r * ldy + c];"),
    "f32_block_one_short": ("for (int64_t c = c0; c < c1; c++) {\n                float a = fabsf(y",
                            "for (int64_t c = c0; c < c1 - 1; c++) {\n                float a = fabsf(y"),
}


def test_real_oracle_passes_every_pin():
    assert all(p() for p in PINS)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    a, b = MUTANTS[name]
    src = orc.source()
    assert src.count(a) >= 1, name
    path = orc.build_variant(src.replace(a, b), "mutant_" + name)
    with orc.using_library(path):
        caught = [p.__name__ for p in PINS if not p()]
    assert caught, f"planted mistake {name} passed every pin"
