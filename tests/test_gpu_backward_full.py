"""The backward pass of the Llama-3.1-8B MLP under the hybrid delayed-scaling
recipe at full size, as the benchmark runs it: per linear (up-projection
4096 -> 14336 and down-projection 14336 -> 4096, M = 8192 tokens), sixteen
steps of dY = 1e-3 * StudentT(3) (seed 100 + t) quantized to E5M2 with the
scale built from the earlier steps' amax history (length 1024, margin 0,
"max"), X and W quantized to E4M3 per tensor ("Infraestructura de
Entrenamiento FP8", introl.com: "Transformer Engine: la base de software";
"Estrategias de escalado y estabilidad").

Every step: all quantized bytes, the amax, the history, the head and the
next scale are compared with the oracle bit for bit.  At steps 0 and 15 the
two products dgrad dX = dY W (MN-major B) and wgrad dW = dY^T X (both
operands MN-major, the whole K accumulated in TMEM and scaled once) are
compared with the oracle on one sampled row per 128-row block and one
sampled column per 256-column block (every output tile is sampled)."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import dev, dev_bf16, f32_bits, host, par_gemm, par_quantize_tensor, stratified

pytestmark = pytest.mark.gpu
REL = 1e-5
M, STEPS, L = 8192, 16, 1024
GEMM_STEPS = (0, STEPS - 1)


def _check(y, y_ref, yabs, out, what):
    bad = orc.check_f32(y, y_ref, yabs, REL) if out == fp8.OUT_F32 else \
        orc.check_bf16(y.view(np.uint16), y_ref, yabs, REL)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; first {i}: "
                             f"got {y[i]} ref {y_ref[i]} abs {yabs[i]}")


def _delayed_e4m3(bits):
    """X or W under its own E4M3 delayed state, as the forward leaves it: one
    step measures its amax, the next quantizes with amax / 448."""
    st = orc.DelayedState(L, orc.E4M3, 0)
    _, amax = par_quantize_tensor(orc, bits, orc.E4M3, float(st.scale[0]))
    st.update(amax)
    q, _ = par_quantize_tensor(orc, bits, orc.E4M3, float(st.scale[0]))
    return q, st.scale.copy()


@pytest.mark.parametrize("name,n_out,k_in", [("up", 14336, 4096), ("down", 4096, 14336)])
def test_mlp_backward_delayed_16_steps_full_size(name, n_out, k_in):
    import torch
    x = inputs.activations(M, k_in, seed=1000 + k_in)
    w = inputs.gaussian((n_out, k_in), 0.02, seed=2000 + n_out)
    qx, sx = _delayed_e4m3(x)
    qw, sw = _delayed_e4m3(w)
    E4, E5, T = fp8.E4M3, fp8.E5M2, fp8.GRAN_TENSOR
    qx_d, qw_d = dev(qx), dev(qw)
    sx_d, sw_d = dev(sx), dev(sw)
    B_dg = fp8.operand(qw_d, sw_d, E4, T, transposed=True)          # W^T: logical [k_in][n_out]
    B_wg = fp8.operand(qx_d, sx_d, E4, T, transposed=True)          # X^T: logical [k_in][M]
    B_dg_o = orc.operand(qw, orc.E4M3, orc.GRAN_TENSOR, sw, transposed=True)
    B_wg_o = orc.operand(qx, orc.E4M3, orc.GRAN_TENSOR, sx, transposed=True)
    rng = np.random.default_rng(n_out)
    dg_rows, dg_cols = stratified(M, 128, rng), stratified(k_in, 256, rng, extra=(k_in - 8,))
    wg_rows, wg_cols = stratified(n_out, 128, rng), stratified(k_in, 256, rng, extra=(k_in - 8,))

    ref = orc.DelayedState(L, orc.E5M2, 0)
    st = fp8.DelayedScaling(L, fp8.E5M2, 0)
    qdy = torch.empty((M, n_out), dtype=torch.uint8, device="cuda")
    dx = torch.empty((M, k_in), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((n_out, k_in), dtype=torch.float32, device="cuda")
    with ThreadPoolExecutor(max_workers=4) as gen:
        dys = [gen.submit(inputs.student_t, (M, n_out), 3.0, 1e-3, 100 + t) for t in range(STEPS)]
        for t in range(STEPS):
            dy = dys[t].result()
            dys[t] = None
            s_used = float(ref.scale[0])
            q_ref, amax_ref = par_quantize_tensor(orc, dy, orc.E5M2, s_used)
            ref.update(amax_ref)
            st.quantize(dev_bf16(dy), q=qdy)
            del dy
            assert f32_bits(host(st.scale))[0] == f32_bits([s_used])[0], (name, t)
            assert np.array_equal(host(qdy), q_ref), (name, t, "codes")
            assert f32_bits(host(st.amax))[0] == f32_bits([amax_ref])[0], (name, t, "amax")
            if t in GEMM_STEPS:
                # this step's products dequantize dY with the scale it was quantized with
                A_dg = fp8.operand(qdy, st.scale, E5, T)                       # [M][n_out]
                A_wg = fp8.operand(qdy, st.scale, E5, T, transposed=True)      # dY^T: [n_out][M]
                fp8.fp8_block_gemm(A_dg, B_dg, M, k_in, n_out, fp8.OUT_BF16, y=dx)
                fp8.fp8_block_gemm(A_wg, B_wg, n_out, k_in, M, fp8.OUT_F32, y=dw)
                fp8.device_status()
                sd = np.float32([s_used])
                A_dg_o = orc.operand(q_ref, orc.E5M2, orc.GRAN_TENSOR, sd)
                A_wg_o = orc.operand(q_ref, orc.E5M2, orc.GRAN_TENSOR, sd, transposed=True)
                y_ref, yabs = par_gemm(orc, M, k_in, n_out, A_dg_o, B_dg_o, dg_rows, dg_cols)
                _check(host(dx)[np.ix_(dg_rows, dg_cols)], y_ref, yabs, fp8.OUT_BF16, f"{name} dgrad step {t}")
                y_ref, yabs = par_gemm(orc, n_out, k_in, M, A_wg_o, B_wg_o, wg_rows, wg_cols)
                _check(host(dw)[np.ix_(wg_rows, wg_cols)], y_ref, yabs, fp8.OUT_F32, f"{name} wgrad step {t}")
            st.update()
            assert np.array_equal(f32_bits(host(st.history)), f32_bits(ref.history)), (name, t, "history")
            assert int(host(st.head)[0]) == int(ref.head[0]), (name, t, "head")
            assert f32_bits(host(st.scale))[0] == f32_bits(ref.scale)[0], (name, t, "scale")
