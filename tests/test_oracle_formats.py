"""Pins of the oracle's FP8 formats and encoder against things other than itself.

- the closed-form facts the pages and the method statement print (golden file);
- code counts implied by the two layouts;
- PyTorch's and ml_dtypes' float8 types used as black-box decoders;
- a brute-force nearest-code search over the decoded table (an independent
  encoder) on a dense sweep of fp32 bit patterns;
- the round-to-nearest-even ties at every midpoint and the saturation rule.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMTS = {"e4m3": orc.E4M3, "e5m2": orc.E5M2}
TORCH_T = {orc.E4M3: torch.float8_e4m3fn, orc.E5M2: torch.float8_e5m2}


def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split(None, 3)


def test_golden_format_facts():
    n = 0
    for fmt, code, value, _src in _golden_rows("fp8_format_facts.txt"):
        got = orc.decode(int(code, 16), FMTS[fmt])
        want = float(value)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (fmt, code)
        n += 1
    assert n >= 14


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_code_counts(fmt):
    t = orc.decode_table(fmt)
    nan = np.isnan(t).sum()
    inf = np.isinf(t).sum()
    if fmt == orc.E4M3:
        assert (nan, inf) == (2, 0)            # S.1111.111 only
        assert np.nanmax(t) == 448.0
    else:
        assert (nan, inf) == (6, 2)            # exponent 31: 2 infinities, 6 NaNs
        assert np.nanmax(t[np.isfinite(t)]) == 57344.0
    # positive codes strictly increasing up to the largest finite code
    pos = t[:128]
    fin = pos[np.isfinite(pos)]
    assert np.all(np.diff(fin) > 0)
    # negative half mirrors the positive half
    assert np.array_equal(np.nan_to_num(t[128:], nan=7.0), -np.nan_to_num(t[:128], nan=-7.0))


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_decode_matches_torch(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(TORCH_T[fmt]).to(torch.float64).numpy()
    got = orc.decode_table(fmt)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_decode_matches_ml_dtypes(fmt):
    mld = pytest.importorskip("ml_dtypes")
    t = mld.float8_e4m3fn if fmt == orc.E4M3 else mld.float8_e5m2
    ref = np.arange(256, dtype=np.uint8).view(t).astype(np.float64)
    got = orc.decode_table(fmt)
    m = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[m], got[m])


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_roundtrip_every_code(fmt):
    t = orc.decode_table(fmt)
    for c in range(256):
        v = t[c]
        if np.isnan(v):
            continue
        got = orc.encode(float(v), fmt)
        if np.isinf(v):   # infinities saturate to the largest finite code
            assert got == (c & 0x80) | 0x7B
        else:
            assert got == c, (fmt, hex(c), v, hex(got))


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_ties_to_even_and_neighbours(fmt):
    t = orc.decode_table(fmt)
    maxcode = 0x7E if fmt == orc.E4M3 else 0x7B
    for c in range(0, maxcode):
        lo, hi = t[c], t[c + 1]
        mid = (lo + hi) / 2                      # exactly representable in fp32 here
        assert float(np.float32(mid)) == mid
        even = c if c % 2 == 0 else c + 1
        assert orc.encode(mid, fmt) == even, (hex(c), mid)
        assert orc.encode(-mid, fmt) == 0x80 | even
        above = float(np.nextafter(np.float32(mid), np.float32(np.inf)))
        below = float(np.nextafter(np.float32(mid), np.float32(-np.inf)))
        assert orc.encode(above, fmt) == c + 1
        assert orc.encode(below, fmt) == c


def test_saturation_and_specials():
    e4, e5 = orc.E4M3, orc.E5M2
    assert orc.encode(464.0, e4) == 0x7E           # tie between 448 and (absent) 480 -> even
    assert orc.encode(470.0, e4) == 0x7E           # rounds past 448 -> saturates
    assert orc.encode(1e30, e4) == 0x7E
    assert orc.encode(-1e30, e4) == 0xFE
    assert orc.encode(float("inf"), e4) == 0x7E
    assert orc.encode(float("-inf"), e4) == 0xFE
    assert orc.encode(61440.0, e5) == 0x7B          # tie 57344/65536 -> 65536 -> saturates
    assert orc.encode(float("inf"), e5) == 0x7B
    assert orc.encode(-0.0, e4) == 0x80
    assert orc.encode(-1e-30, e4) == 0x80
    assert orc.encode(0.0, e5) == 0x00
    assert orc.encode(2.0 ** -10, e4) == 0x00      # half of the smallest subnormal -> even (0)
    assert orc.encode(3 * 2.0 ** -10, e4) == 0x02  # 1.5 * 2^-9 -> tie -> 2 * 2^-9
    assert orc.encode(float("nan"), e4) == 0x7F


def _brute_force_encode(v: np.ndarray, fmt: int) -> np.ndarray:
    """Independent encoder: nearest entry of the decoded table, ties to the
    even code, magnitudes beyond the largest finite value saturate."""
    t = orc.decode_table(fmt)
    maxcode = 0x7E if fmt == orc.E4M3 else 0x7B
    mags = t[: maxcode + 1]                      # increasing, 0 .. fmax
    a = np.abs(v.astype(np.float64))
    hi = np.searchsorted(mags, a, side="left")   # first index with mags >= a
    hi_c = np.clip(hi, 0, maxcode)
    lo_c = np.clip(hi - 1, 0, maxcode)
    d_hi = np.abs(mags[hi_c] - a)
    d_lo = np.abs(a - mags[lo_c])
    pick = np.where(d_lo < d_hi, lo_c, hi_c)
    tie = (d_lo == d_hi) & (lo_c != hi_c)
    pick = np.where(tie, np.where(lo_c % 2 == 0, lo_c, hi_c), pick)
    # beyond fmax: nearest in an unbounded format would be the next binade's
    # first value or more -> saturate; within half a step above fmax the
    # nearest is fmax itself (handled by the clip above).
    pick = np.where(a >= mags[-1], maxcode, pick)
    sign = np.signbit(v).astype(np.int64) << 7
    return (pick | sign).astype(np.uint8)


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_encode_sweep_vs_brute_force(fmt):
    # every 61st fp32 bit pattern of the finite range, both signs (~70M values),
    # plus every pattern in the binades around the subnormal/normal boundary.
    step = 61
    pats = np.arange(0, 0x7F800000, step, dtype=np.uint32)
    lo_e = 0x3A000000 if fmt == orc.E4M3 else 0x36000000     # ~2^-11 / ~2^-19
    dense = np.arange(lo_e, lo_e + (3 << 23), 1, dtype=np.uint32)
    chunk = 1 << 22
    for block in (pats, dense):
        for sgn in (0, 0x80000000):
            for i in range(0, block.size, chunk):
                v = (block[i:i + chunk] | np.uint32(sgn)).view(np.float32)
                got = orc.encode_array(v, fmt)
                want = _brute_force_encode(v, fmt)
                bad = np.nonzero(got != want)[0]
                assert bad.size == 0, (fmt, v[bad[:5]], got[bad[:5]], want[bad[:5]])


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_encode_matches_torch_cast_in_range(fmt):
    # torch's float32 -> float8 cast rounds to nearest-even; it does not
    # saturate, so compare only where no overflow can occur.
    rng = np.random.default_rng(7)
    lim = 464.0 if fmt == orc.E4M3 else 61440.0
    v = np.concatenate([
        rng.uniform(-lim, lim, 200000),
        rng.standard_normal(200000) * 10.0 ** rng.uniform(-12, 4, 200000),
    ]).astype(np.float32)
    v = v[np.abs(v) < lim]
    ref = torch.from_numpy(v).to(TORCH_T[fmt]).view(torch.uint8).numpy()
    got = orc.encode_array(v, fmt)
    assert np.array_equal(ref, got)
