"""Device-side failure detection without faulting the GPU: the bounded
mbarrier wait used by every GEMM role gives up on a barrier nothing arrives
at, the status word reports it, and the context keeps working."""
import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import dev_bf16, host

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    fp8.device_status()                              # clean slate
    assert fp8.selftest_wait_timeout(limit_ms=200)   # the wait gave up
    with pytest.raises(fp8.Fp8bsError) as e:
        fp8.device_status()
    assert e.value.code == -5                        # FP8BS_ERR_DEVICE_TIMEOUT
    fp8.device_status()                              # the record was cleared
    # the context is usable: a quantize + GEMM still matches the oracle
    x = inputs.activations(128, 256, seed=5)
    w = inputs.gaussian((256, 256), 0.02, seed=6)
    qx, sx = fp8.fp8_quantize_1x128(dev_bf16(x))
    qw, sw = fp8.fp8_quantize_128x128(dev_bf16(w))
    y = fp8.fp8_block_gemm(fp8.operand(qx, sx), fp8.operand(qw, sw, gran=fp8.GRAN_128x128),
                           128, 256, 256, fp8.OUT_F32)
    rqx, rsx = orc.quantize_1x128(x)
    rqw, rsw = orc.quantize_128x128(w)
    assert np.array_equal(host(qx), rqx)
    y_ref, yabs = orc.gemm(128, 256, 256, orc.operand(rqx, orc.E4M3, orc.GRAN_1x128, rsx),
                           orc.operand(rqw, orc.E4M3, orc.GRAN_128x128, rsw))
    assert not orc.check_f32(host(y), y_ref, yabs).any()
    fp8.device_status()
