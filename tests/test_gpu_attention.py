"""Parity of the FP8 attention (FP8 KV cache) with the oracle.  The kernel
rounds the softmax numerators P to E4M3, so outputs are accepted under the
bound derived from that rounding (oracle.check_attention_bf16); where every
score of a row is equal (P = 1, exact in E4M3) the output must be the plain
mean of the visible values."""
import numpy as np
import pytest

import block_scaled_gemm_quantize_gb300 as fp8
import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from helpers import dev, host, stratified

pytestmark = pytest.mark.gpu
SCALE = 128 ** -0.5


def _inputs(S_q, S_k, hq, hkv, seed, zero_k=False, v_tile_gain=None):
    """v_tile_gain: per 128-key tile factors applied to V (0 = a tile of
    zeros), or "equal": each tile's first key set to 8 in every element, so
    every V tile of a head gets the same scale."""
    q = inputs.gaussian((S_q, hq * 128), 1.0, seed=seed)
    k = inputs.gaussian((max(S_k, 1), hkv * 128), 1.0, seed=seed + 1)[:S_k]
    v = inputs.gaussian((max(S_k, 1), hkv * 128), 1.0, seed=seed + 2)[:S_k]
    if v_tile_gain is not None and S_k:
        vf = inputs.bits_to_f32(v).astype(np.float64)
        if isinstance(v_tile_gain, str):
            vf[::128] = 8.0
        else:
            vf *= np.repeat(np.asarray(v_tile_gain, np.float64), 128)[:S_k, None]
        v = inputs.bf16_bits(vf.astype(np.float32))
    qq, sq = orc.quantize_1x128(q)
    kq, sk = orc.quantize_128x128(k) if S_k else (np.zeros((0, hkv * 128), np.uint8), np.ones((1, hkv), np.float32))
    vq, sv = orc.quantize_128x128(v) if S_k else (np.zeros((0, hkv * 128), np.uint8), np.ones((1, hkv), np.float32))
    if zero_k:
        kq = np.zeros_like(kq)
    return qq, sq, kq, sk, vq, sv


def _run(S_q, S_k, hq, hkv, causal, arrs):
    import torch
    qq, sq, kq, sk, vq, sv = arrs
    Kd = dev(kq) if S_k else torch.zeros((16, hkv * 128), dtype=torch.uint8, device="cuda")
    Vd = dev(vq) if S_k else torch.zeros((16, hkv * 128), dtype=torch.uint8, device="cuda")
    Q = fp8.attn_input(dev(qq), dev(sq))
    K = fp8.attn_input(Kd, dev(sk))
    V = fp8.attn_input(Vd, dev(sv))
    o = fp8.fp8_attention_fwd(Q, K, V, S_q, S_k, hq, hkv, causal, SCALE)
    fp8.device_status()
    return host(o).reshape(S_q * hq, 128)      # rows ordered (token, head)


def _check(o_bits, ref):
    o, oap, oav = ref
    bad = orc.check_attention_bf16(o_bits, o, oap, oav)
    assert not bad.any(), f"{int(bad.sum())}/{bad.size} outside the P-rounding bound"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S_q,S_k,hq,hkv", [(300, 384, 4, 2), (256, 256, 4, 1), (200, 456, 2, 2), (130, 130, 8, 8),
                                             # more queries than keys: causal rows below
                                             # seq_q - seq_k see no key (whole tiles of them)
                                             (400, 200, 2, 1), (300, 130, 4, 2)])
def test_attention_small(causal, S_q, S_k, hq, hkv):
    arrs = _inputs(S_q, S_k, hq, hkv, seed=S_q + S_k)
    o_bits = _run(S_q, S_k, hq, hkv, causal, arrs)
    _check(o_bits, orc.attention(S_q, S_k, hq, hkv, causal, SCALE, *arrs))
    if causal and S_q > S_k:   # rows that see no key are 0
        assert np.all(o_bits[: (S_q - S_k) * hq] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_more_than_32_key_tiles(causal):
    """Keys spanning 33 tiles of 128 plus a ragged one: the per-tile K and V
    scales come from a window of 32 tiles that is reloaded past tile 31."""
    S_q, S_k, hq, hkv = 200, 4300, 2, 1
    arrs = _inputs(S_q, S_k, hq, hkv, seed=33)
    o_bits = _run(S_q, S_k, hq, hkv, causal, arrs)
    _check(o_bits, orc.attention(S_q, S_k, hq, hkv, causal, SCALE, *arrs))


def test_attention_equal_scores_give_the_mean_of_the_visible_values():
    """All keys equal and every V tile of the head at the same scale: each
    visible P is exactly 448 in E4M3 (P is scaled by its tile's V scale over
    the head's largest, here 1), so the output is the plain mean."""
    import torch
    S, hq, hkv = 384, 2, 1
    arrs = _inputs(S, S, hq, hkv, seed=7, zero_k=True, v_tile_gain="equal")
    assert np.all(arrs[5] == arrs[5][0])
    o_bits = _run(S, S, hq, hkv, True, arrs)
    o = torch.from_numpy(o_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ref, _, _ = orc.attention(S, S, hq, hkv, True, SCALE, *arrs)
    # P = 1 exactly, so only fp32 accumulation and the bf16 store round the mean
    assert np.all(np.abs(o - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max())


def test_attention_without_keys_gives_zeros():
    arrs = _inputs(130, 0, 2, 1, seed=9)
    o_bits = _run(130, 0, 2, 1, False, arrs)
    assert np.all(o_bits == 0)


def test_attention_llama31_8b_prefill_sampled():
    """Llama-3.1-8B attention prefill (8192 tokens, 32 query heads, 8 KV heads,
    causal) at full size, as the attention benchmark runs it; sampled rows."""
    S, hq, hkv = 8192, 32, 8
    arrs = _inputs(S, S, hq, hkv, seed=21)
    o_bits = _run(S, S, hq, hkv, True, arrs)
    rng = np.random.default_rng(3)
    rows = stratified(S, 512, rng, extra=(1, 127, 128, 4095))
    heads = rng.integers(0, hq, rows.size)
    ref = orc.attention(S, S, hq, hkv, True, SCALE, *arrs, rows=rows, heads=heads)
    _check(o_bits[rows * hq + heads], ref)


@pytest.mark.parametrize("zero_scale", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_v_tiles_with_very_different_scales_and_a_zero_tile(causal, zero_scale):
    """V tiles scaled by 1 .. 2^-12 and one tile of zeros (its scale as the
    quantizer gives it, 1, which then is the head's largest; or 0): P is
    quantized after the factor sv_t / (largest V scale of the head), so
    small-scale tiles lose precision only in the subnormal range the bound
    allows; the zero tile contributes nothing (its keys still count in the
    row sum)."""
    S_q, S_k, hq, hkv = 256, 896, 2, 2
    gains = [1.0, 2.0 ** -4, 0.0, 2.0 ** -12, 0.5, 2.0 ** -8, 1.0]
    arrs = _inputs(S_q, S_k, hq, hkv, seed=91, v_tile_gain=gains)
    if zero_scale:
        arrs[5][2] = 0.0
    o_bits = _run(S_q, S_k, hq, hkv, causal, arrs)
    _check(o_bits, orc.attention(S_q, S_k, hq, hkv, causal, SCALE, *arrs))
