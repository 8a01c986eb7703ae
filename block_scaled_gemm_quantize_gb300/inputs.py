"""Seeded synthetic inputs shaped like the FP8-training pages' workloads.

This module holds no FP8 arithmetic: it only draws random numbers, rounds
them to bf16 (the layer's input dtype) and describes the workloads.  Both the
CUDA path's tests and the oracle take their inputs from here.

The pages measure Llama-2 7B, Llama 3.1 8B and Qwen3-30B models (introl.com
"El panorama de la precision numerica"; hotbookzone.com "El avance tecnico"
and "Ganancias de rendimiento en el mundo real"); no weights or data exist
here, so these shapes and distributions stand in for those models' linear
layers.
"""
from __future__ import annotations

import numpy as np


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even), returned as uint16 bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def gaussian(shape, std: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def activations(M: int, K: int, seed: int, outlier_frac: float = 0.01,
                outlier_gain: float = 20.0) -> np.ndarray:
    """N(0,1) activations with round(frac*K) seeded outlier channels x gain."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    n_out = int(round(outlier_frac * K))
    if n_out:
        cols = rng.choice(K, size=n_out, replace=False)
        x[:, cols] *= np.float32(outlier_gain)
    return bf16_bits(x)


def student_t(shape, nu: float, scale: float, seed: int) -> np.ndarray:
    """Heavy-tailed gradients: scale * StudentT(nu) (scale is the t scale)."""
    rng = np.random.default_rng(seed)
    return bf16_bits((rng.standard_t(nu, size=shape) * scale).astype(np.float32))


def moe_routing(tokens: int, experts: int, topk: int, zipf_a: float, seed: int):
    """Top-k distinct experts per token drawn with p ~ rank^-a over a seeded
    rank->expert permutation.  Returns (loads [experts], offsets [experts+1])
    for the expert-sorted row order."""
    rng = np.random.default_rng(seed)
    p = np.arange(1, experts + 1, dtype=np.float64) ** (-zipf_a)
    p /= p.sum()
    perm = rng.permutation(experts)
    loads = np.zeros(experts, dtype=np.int64)
    for _ in range(tokens):
        ranks = rng.choice(experts, size=topk, replace=False, p=p)
        loads[perm[ranks]] += 1
    offsets = np.zeros(experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(loads)
    return loads, offsets


# ------------------------------------------------------------- workloads
# (name, M, N, K) per linear; X is [M, K], W is [N, K], Y = X W^T is [M, N].
LLAMA2_7B_FPROP = dict(
    name="llama2-7b-fprop", M=4096, scale_mode="pow2",
    linears=[("qkv", 12288, 4096), ("o", 4096, 4096), ("gate_up", 22016, 4096),
             ("down", 4096, 11008)])
LLAMA31_8B_FPROP = dict(
    name="llama3.1-8b-fprop", M=8192, scale_mode="fp32",
    linears=[("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 28672, 4096),
             ("down", 4096, 14336)])
TINY_FPROP = dict(name="tiny-fprop", M=256, scale_mode="fp32", linears=[("tiny", 256, 512)])
LLAMA31_8B_MLP_BWD = dict(
    name="llama3.1-8b-mlp-bwd", M=8192, steps=16, history_len=1024, margin=0,
    # (name, N_out, K_in): up-projection 4096->14336, down-projection 14336->4096
    linears=[("up", 14336, 4096), ("down", 4096, 14336)], dy_scale=1e-3, dy_nu=3.0)
QWEN3_30B_MOE = dict(
    name="qwen3-30b-a3b-moe", tokens=8192, hidden=2048, experts=128, topk=8, zipf_a=1.1,
    gate_up_n=1536, down_k=768)

# An MLP block as a chain of two FP8 linears whose intermediate never leaves
# FP8: gate/up product with a SwiGLU + 1x128-quantizing epilogue, then the
# down product on those codes (dense Llama-3.1-8B MLP; Qwen3-30B-A3B experts).
LLAMA31_8B_MLP_FUSED = dict(name="llama3.1-8b-mlp-fused", M=8192, hidden=4096,
                            intermediate=14336, scale_mode="fp32")
QWEN3_30B_MOE_FUSED = dict(name="qwen3-30b-a3b-moe-fused", tokens=8192, hidden=2048, experts=128,
                           topk=8, zipf_a=1.1, intermediate=768, scale_mode="fp32")

# The same MLP backward under the block recipe: dY and X quantized per 1x128
# tile along the contraction of each product (row-wise for dgrad, column-wise
# transposed copies for wgrad), W per 128x128 tile, E4M3 throughout.
LLAMA31_8B_MLP_BWD_BLOCK = dict(
    name="llama3.1-8b-mlp-bwd-blockwise", M=8192, scale_mode="fp32",
    linears=[("up", 14336, 4096), ("down", 4096, 14336)], dy_scale=1e-3, dy_nu=3.0)

# The Llama-3.1-8B fprop linears in MXFP8 (1x32 blocks, E8M0 scales) on
# both operands, the block-scaling format Blackwell's tensor cores apply.
LLAMA31_8B_FPROP_MX = dict(
    name="llama3.1-8b-fprop-mxfp8", M=8192, scale_mode="mx",
    linears=[("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 28672, 4096),
             ("down", 4096, 14336)])

# Llama-3.1-8B attention prefill over an FP8 KV cache: 8192 tokens, 32 query
# heads sharing 8 key/value heads, head_dim 128, causal.
LLAMA31_8B_ATTN = dict(name="llama3.1-8b-attn-fp8", seq=8192, heads_q=32, heads_kv=8, causal=True)
