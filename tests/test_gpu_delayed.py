"""Parity of per-tensor delayed scaling (quantizer + amax history) with the
oracle, step by step: codes, amax, history, head and scale bit-exact."""
import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import dev_bf16, f32_bits, host

pytestmark = pytest.mark.gpu


def _run(shape, steps, L, fmt, margin, scale_fn):
    ref = orc.DelayedState(L, fmt, margin)
    st = fp8.DelayedScaling(L, fmt, margin)
    for t in range(steps):
        x = inputs.student_t(shape, 3.0, scale_fn(t), seed=100 + t)
        q_ref, amax_ref = ref.step(x)
        q = st.quantize(dev_bf16(x), update=True)
        assert np.array_equal(host(q), q_ref), t
        assert f32_bits(host(st.amax))[0] == f32_bits([amax_ref])[0], t
        assert np.array_equal(f32_bits(host(st.history)), f32_bits(ref.history)), t
        assert int(host(st.head)[0]) == int(ref.head[0])
        assert f32_bits(host(st.scale))[0] == f32_bits(ref.scale)[0], t
    return st, ref


@pytest.mark.parametrize("fmt", [fp8.E5M2, fp8.E4M3])
def test_delayed_16_steps(fmt):
    _run((64, 1024), 16, 1024, fmt, 0, lambda t: 1e-3 * (1 + (t % 5)))


def test_delayed_wrap_margin_ragged():
    # history of 4 wraps; margin 1; numel not a multiple of 8 (ragged tail)
    _run((1, 1003), 9, 4, fp8.E5M2, 1, lambda t: 1e-3 * (9 - t))


def test_delayed_save_restore():
    st, ref = _run((32, 512), 5, 8, fp8.E5M2, 0, lambda t: 1e-3)
    sd = st.state_dict()
    st2 = fp8.DelayedScaling(8, fp8.E5M2)
    st2.load_state_dict(sd)
    x = inputs.student_t((32, 512), 3.0, 1e-3, seed=999)
    q_ref, _ = ref.step(x)
    assert np.array_equal(host(st2.quantize(dev_bf16(x), update=True)), q_ref)
