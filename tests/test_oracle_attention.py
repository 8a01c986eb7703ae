"""Pins of the FP8 attention oracle: numpy softmax attention on the
dequantized tensors (PyTorch float8 decode), closed-form cases (the first
causal row sees one key; equal scores average the values), and the acceptance
rule against a numpy evaluation that rounds P to E4M3 as the kernel does."""
import numpy as np
import pytest
import torch

import oracle as orc
from block_scaled_gemm_quantize_gb300 import inputs
from test_oracle_fused import _nearest_code


def _deq(q, tt=torch.float8_e4m3fn):
    return torch.from_numpy(np.ascontiguousarray(q)).view(tt).to(torch.float64).numpy()


def _case(S_q, S_k, hq, hkv, seed):
    x = inputs.activations(S_q, hq * 128, seed=seed)
    k = inputs.activations(S_k, hkv * 128, seed=seed + 1)
    v = inputs.gaussian((S_k, hkv * 128), 1.0, seed=seed + 2)
    qq, sq = orc.quantize_1x128(x)
    kq, sk = orc.quantize_128x128(k)
    vq, sv = orc.quantize_128x128(v)
    Q = _deq(qq).reshape(S_q, hq, 128) * sq.T[:, :, None]
    K = _deq(kq).reshape(S_k, hkv, 128) * np.repeat(sk, 128, axis=0)[:S_k, :, None]
    V = _deq(vq).reshape(S_k, hkv, 128) * np.repeat(sv, 128, axis=0)[:S_k, :, None]
    return (qq, sq, kq, sk, vq, sv), (Q, K, V)


def _numpy_attention(Q, K, V, causal, scale):
    S_q, hq, _ = Q.shape
    S_k, hkv, _ = K.shape
    out = np.zeros_like(Q)
    for h in range(hq):
        g = h // (hq // hkv)
        s = Q[:, h] @ K[:, g].T * scale
        if causal:
            mask = np.arange(S_k)[None, :] > (np.arange(S_q)[:, None] + S_k - S_q)
            s = np.where(mask, -np.inf, s)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        out[:, h] = (p / p.sum(axis=1, keepdims=True)) @ V[:, g]
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S_q,S_k,hq,hkv", [(200, 200, 4, 2), (130, 300, 2, 1), (256, 256, 4, 4)])
def test_attention_matches_numpy(causal, S_q, S_k, hq, hkv):
    (qq, sq, kq, sk, vq, sv), (Q, K, V) = _case(S_q, S_k, hq, hkv, seed=31)
    scale = 1.0 / np.sqrt(128.0)
    o, _, _ = orc.attention(S_q, S_k, hq, hkv, causal, scale, qq, sq, kq, sk, vq, sv)
    ref = _numpy_attention(Q, K, V, causal, scale).reshape(S_q * hq, 128)
    assert np.allclose(o, ref, rtol=1e-10, atol=1e-12)


def test_first_causal_row_sees_one_key_and_equal_scores_average():
    (qq, sq, kq, sk, vq, sv), (Q, K, V) = _case(128, 128, 2, 1, seed=41)
    o, _, _ = orc.attention(128, 128, 2, 1, True, 0.1, qq, sq, kq, sk, vq, sv,
                            rows=[0, 0], heads=[0, 1])
    assert np.array_equal(o[0], V[0, 0]) and np.array_equal(o[1], V[0, 0])
    kz = np.zeros_like(kq)                       # all keys equal: P = 1 for every visible key
    o2, _, _ = orc.attention(128, 128, 2, 1, True, 0.1, qq, sq, kz, sk, vq, sv, rows=[5, 77], heads=[1, 0])
    assert np.allclose(o2[0], V[:6, 0].mean(axis=0), rtol=1e-13)
    assert np.allclose(o2[1], V[:78, 0].mean(axis=0), rtol=1e-13)


def test_acceptance_rule_covers_e4m3_rounding_of_p_and_rejects_a_wrong_mask():
    S, hq, hkv = 256, 2, 1
    (qq, sq, kq, sk, vq, sv), (Q, K, V) = _case(S, S, hq, hkv, seed=51)
    scale = 1.0 / np.sqrt(128.0)
    o, oap, oav = orc.attention(S, S, hq, hkv, True, scale, qq, sq, kq, sk, vq, sv)
    # numpy evaluation with P rounded to E4M3 at scale 1/448 (l from unrounded P)
    sim = np.zeros((S, hq, 128))
    for h in range(hq):
        s = Q[:, h] @ K[:, 0].T * scale
        s = np.where(np.arange(S)[None, :] > np.arange(S)[:, None], -np.inf, s)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        pq = _deq(_nearest_code((p * 448.0).astype(np.float32), orc.E4M3)) / 448.0
        sim[:, h] = (pq @ V[:, 0]) / p.sum(axis=1, keepdims=True)
    bits = torch.from_numpy(sim.reshape(S * hq, 128)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert not orc.check_attention_bf16(bits, o, oap, oav).any()
    # the same evaluation without the causal mask is rejected
    wrong = np.zeros((S, hq, 128))
    for h in range(hq):
        s = Q[:, h] @ K[:, 0].T * scale
        p = np.exp(s - s.max(axis=1, keepdims=True))
        wrong[:, h] = (p @ V[:, 0]) / p.sum(axis=1, keepdims=True)
    wb = torch.from_numpy(wrong.reshape(S * hq, 128)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert orc.check_attention_bf16(wb, o, oap, oav).mean() > 0.3


def test_tolerance_terms_match_their_definitions():
    """oap = sum_j P |deqV| / l and oav = sum_j |V code| svm / l (svm: the
    head's largest V tile scale), against numpy on the dequantized tensors."""
    S, hq, hkv = 200, 2, 1
    (qq, sq, kq, sk, vq, sv), (Q, K, V) = _case(S, S, hq, hkv, seed=61)
    scale = 1.0 / np.sqrt(128.0)
    _, oap, oav = orc.attention(S, S, hq, hkv, True, scale, qq, sq, kq, sk, vq, sv)
    codes = _deq(vq).reshape(S, hkv, 128)
    svm = float(sv[:, 0].max())
    for h in range(hq):
        s = Q[:, h] @ K[:, 0].T * scale
        s = np.where(np.arange(S)[None, :] > np.arange(S)[:, None], -np.inf, s)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        l = p.sum(axis=1, keepdims=True)
        rows = np.arange(S) * hq + h
        assert np.allclose(oap[rows], (p @ np.abs(V[:, 0])) / l, rtol=1e-12)
        vis = (np.arange(S)[None, :] <= np.arange(S)[:, None]).astype(np.float64)
        assert np.allclose(oav[rows], (vis @ np.abs(codes[:, 0])) * svm / l, rtol=1e-12)


def test_acceptance_rule_covers_p_rounded_after_the_v_scale_ratio():
    """V tiles whose scales differ by up to 2^10: a numpy evaluation that
    rounds P * sv_t / svm to E4M3 at 1/448 (and reads it back times
    svm / sv_t, l from unrounded P) stays inside the rule."""
    S, hq, hkv = 384, 2, 1
    x = inputs.activations(S, hq * 128, seed=71)
    k = inputs.activations(S, hkv * 128, seed=72)
    vf = inputs.bits_to_f32(inputs.gaussian((S, hkv * 128), 1.0, seed=73)).astype(np.float64)
    vf *= np.repeat(2.0 ** np.array([0.0, -6.0, -10.0]), 128)[:, None]
    v = inputs.bf16_bits(vf.astype(np.float32))
    qq, sq = orc.quantize_1x128(x)
    kq, sk = orc.quantize_128x128(k)
    vq, sv = orc.quantize_128x128(v)
    Q = _deq(qq).reshape(S, hq, 128) * sq.T[:, :, None]
    K = _deq(kq).reshape(S, hkv, 128) * np.repeat(sk, 128, axis=0)[:S, :, None]
    V = _deq(vq).reshape(S, hkv, 128) * np.repeat(sv, 128, axis=0)[:S, :, None]
    scale = 1.0 / np.sqrt(128.0)
    o, oap, oav = orc.attention(S, S, hq, hkv, True, scale, qq, sq, kq, sk, vq, sv)
    ratio = np.repeat(sv[:, 0] / sv[:, 0].max(), 128)[:S]
    sim = np.zeros((S, hq, 128))
    for h in range(hq):
        s = Q[:, h] @ K[:, 0].T * scale
        s = np.where(np.arange(S)[None, :] > np.arange(S)[:, None], -np.inf, s)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        pq = _deq(_nearest_code((p * ratio[None, :] * 448.0).astype(np.float32), orc.E4M3)) / 448.0
        sim[:, h] = ((pq / ratio[None, :]) @ V[:, 0]) / p.sum(axis=1, keepdims=True)
    bits = torch.from_numpy(sim.reshape(S * hq, 128)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert not orc.check_attention_bf16(bits, o, oap, oav).any()
