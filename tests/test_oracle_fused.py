"""Pins of the oracle pieces behind the quantized-output product: the 1x128
rule on fp32 input, the SwiGLU gate and its interval bounds, and the
acceptance rule for a quantization of values known only within a tolerance.
Each is tied to something other than itself: the already pinned bf16
quantizer, numpy tile reductions with a brute-force nearest-code search,
scipy's logistic function, closed forms, and dense sampling."""
import numpy as np
import pytest
import torch

import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs


def _nearest_code(v, fmt):
    """Brute force: the code nearest to each fp32 value (ties to the even
    code, saturation at the largest finite code), searched over the table of
    decoded values that PyTorch's float8 types give."""
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


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
@pytest.mark.parametrize("mode", [orc.SCALE_FP32, orc.SCALE_POW2])
def test_f32_rule_reduces_to_bf16_rule_on_bf16_values(fmt, mode):
    x = inputs.activations(33, 384, seed=5)
    q_ref, s_ref = orc.quantize_1x128(x, fmt, mode)
    q, s = orc.quantize_1x128_f32(inputs.bits_to_f32(x), fmt, mode)
    assert np.array_equal(q, q_ref) and np.array_equal(s, s_ref)


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_f32_rule_matches_numpy_tiles_and_brute_force(fmt):
    rng = np.random.default_rng(7)
    y = (rng.standard_normal((17, 256)) * 10.0 ** rng.uniform(-3, 3, (17, 1))).astype(np.float32)
    y[3, :128] = 0.0                                      # a zero block -> scale 1
    q, s = orc.quantize_1x128_f32(y, fmt, orc.SCALE_FP32)
    amax = np.abs(y).reshape(17, 2, 128).max(axis=2)
    fm = np.float32(448.0 if fmt == orc.E4M3 else 57344.0)
    want = np.where(amax == 0, np.float32(1.0), np.maximum((amax / fm).astype(np.float32),
                                                          np.float32(2.0 ** -126)))
    assert np.array_equal(s, want.T.astype(np.float32))
    r = (np.float32(1.0) / np.repeat(want, 128, axis=1)).astype(np.float32)
    assert np.array_equal(q, _nearest_code((y * r).astype(np.float32), fmt))


def test_swiglu_against_scipy_logistic_and_closed_forms():
    from scipy.special import expit
    rng = np.random.default_rng(3)
    g = rng.standard_normal(1000) * 6
    u = rng.standard_normal(1000)
    assert np.allclose(orc.swiglu(g, u), g * expit(g) * u, rtol=1e-14, atol=0)
    # s(ln 3) = 3/4, so silu(ln 3) = 0.75 ln 3; silu(0) = 0; silu(x) -> x and -> 0
    assert abs(orc.swiglu(np.log(3.0), 1.0) - 0.75 * np.log(3.0)) < 1e-15
    assert orc.swiglu(0.0, 5.0) == 0.0
    assert orc.swiglu(800.0, 1.0) == 800.0 and abs(orc.swiglu(-800.0, 1.0)) == 0.0


def test_silu_minimum():
    x = orc.SILU_ARGMIN
    assert -1.2785 < x < -1.2784
    h = 1e-5
    d = (orc.swiglu(x + h, 1.0) - orc.swiglu(x - h, 1.0)) / (2 * h)
    assert abs(d) < 1e-9
    grid = np.linspace(-4, 2, 600001)
    assert orc.swiglu(x, 1.0) <= orc.swiglu(grid, np.ones_like(grid)).min() + 1e-15


def test_silu_range_and_swiglu_bounds_contain_dense_samples():
    rng = np.random.default_rng(11)
    c = rng.uniform(-6, 6, 300)
    w = rng.uniform(0, 2, 300)
    mn, mx = orc.silu_range(c - w, c + w)
    uc, uw = rng.standard_normal(300), rng.uniform(0, 0.5, 300)
    lo, hi = orc.swiglu_bounds(c, w, uc, uw, rel=0.0, rel_g=0.0)
    t = np.linspace(0, 1, 201)
    gs = (c - w)[:, None] + (2 * w)[:, None] * t[None, :]
    sv = orc.swiglu(gs, np.ones_like(gs))
    assert np.all(sv >= mn[:, None] - 1e-12) and np.all(sv <= mx[:, None] + 1e-12)
    assert np.allclose(sv.min(axis=1), mn, atol=1e-4) and np.allclose(sv.max(axis=1), mx, atol=0)
    for us in (uc - uw, uc + uw, uc):
        hv = sv * us[:, None]
        assert np.all(hv >= lo[:, None] - 1e-12) and np.all(hv <= hi[:, None] + 1e-12)


@pytest.mark.parametrize("mode", [orc.SCALE_FP32, orc.SCALE_POW2])
def test_acceptance_exact_intervals_accept_only_the_oracle_result(mode):
    rng = np.random.default_rng(1)
    y = (rng.standard_normal((9, 384)) * 3).astype(np.float32)
    y[2, 128:256] = 0.0
    q, s = orc.quantize_1x128_f32(y, orc.E4M3, mode)
    bs, bc = orc.check_quantized_1x128(q, s, y, y, orc.E4M3, mode)
    assert not bs.any() and not bc.any()
    # one code one step off in value order (away from zero) is rejected
    q2 = q.copy()
    c = int(q2[4, 7])
    q2[4, 7] = c + 1 if (c & 0x7F) < 0x7E else c - 1
    assert orc.check_quantized_1x128(q2, s, y, y, orc.E4M3, mode)[1][4, 7]
    # a scale one ulp (fp32) or one binade (pow2) off is rejected
    s2 = s.copy()
    s2[1, 5] = np.nextafter(s2[1, 5], np.float32(np.inf)) if mode == orc.SCALE_FP32 else s2[1, 5] * 2
    assert orc.check_quantized_1x128(q, s2, y, y, orc.E4M3, mode)[0][1, 5]


def test_acceptance_interval_across_a_rounding_midpoint_accepts_both_codes():
    # a block whose amax is 448 (scale 1, fp32 rule): element 1.0625 lies
    # exactly between the E4M3 codes of 1.0 and 1.125
    y = np.zeros((1, 128), np.float32)
    y[0, 0] = 448.0
    y[0, 1] = 1.0625
    lo = y.astype(np.float64).copy()
    hi = lo.copy()
    lo[0, 1] -= 1e-6
    hi[0, 1] += 1e-6
    s = np.float32([[1.0]])
    for code in (0x38, 0x39):                          # 1.0 and 1.125
        q = orc.encode_array(y, orc.E4M3)
        q[0, 1] = code
        bs, bc = orc.check_quantized_1x128(q, s, lo, hi, orc.E4M3, orc.SCALE_FP32)
        assert not bs.any() and not bc.any()
    q[0, 1] = 0x3A                                     # 1.25: outside
    assert orc.check_quantized_1x128(q, s, lo, hi, orc.E4M3, orc.SCALE_FP32)[1][0, 1]


def test_swiglu_slack_covers_fast_fp32_evaluation():
    """The default slack of swiglu_bounds covers an fp32 evaluation that uses
    a base-2 exponential of the fp32-rounded argument -g log2(e) (the form of
    the fast exponential), simulated here in numpy with the argument rounding
    made explicit and the other steps rounded to fp32."""
    rng = np.random.default_rng(4)
    g = np.concatenate([rng.standard_normal(20000) * 8, rng.uniform(-80, 80, 20000)])
    u = rng.standard_normal(g.size)
    arg = (np.float32(-1.0) * g.astype(np.float32) * np.float32(np.log2(np.e))).astype(np.float32)
    e = np.exp2(arg.astype(np.float64)).astype(np.float32)
    den = (np.float32(1.0) + e).astype(np.float32)
    h = ((g.astype(np.float32) * (np.float32(1.0) / den).astype(np.float32)).astype(np.float32)
         * u.astype(np.float32)).astype(np.float64)
    gr, ur = g.astype(np.float32).astype(np.float64), u.astype(np.float32).astype(np.float64)
    lo, hi = orc.swiglu_bounds(gr, 0.0, ur, 0.0)
    assert np.all((h >= lo) & (h <= hi))
    # and without the slack this evaluation falls outside somewhere
    lo0, hi0 = orc.swiglu_bounds(gr, 0.0, ur, 0.0, rel=0.0, rel_g=0.0)
    assert np.any((h < lo0) | (h > hi0))
