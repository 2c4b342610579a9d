"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws random numbers and rounds them to bf16 (the input
format), and builds the rotary cos/sin tables that the rotary embedding
takes as inputs; it holds none of the NVFP4 arithmetic (no scales, no
quantization, no GEMM) and none of the rotation itself.  Every generator is numpy PCG64 (``default_rng(seed)``) drawing
float32, rounded to bf16 with round-to-nearest-even by torch's CPU cast.
bf16 tensors are returned as numpy ``uint16`` bit patterns.

Shapes follow the 27B-class dense model of the workloads: hidden H=5120,
intermediate I=17408, QKV N=7168 (5120 Q + 2 x 1024 KV), O 5120.
"""
from __future__ import annotations

import numpy as np
import torch

H = 5120
I = 17408
QKV = 7168
NORM_EPS = 1e-6


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(rng: np.random.Generator, shape, mean=0.0, std=1.0) -> np.ndarray:
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return f32_to_bf16_bits(a)


def student_t_outliers(rng: np.random.Generator, shape, df=3.0, channel_frac=0.001, factor=100.0):
    """Student-t(df) activations with round(channel_frac * cols) channels
    (chosen by the rng) scaled by ``factor``."""
    a = rng.standard_t(df, size=shape).astype(np.float32)
    n_out = int(round(channel_frac * shape[-1]))
    ch = rng.choice(shape[-1], size=n_out, replace=False)
    a[..., ch] *= np.float32(factor)
    return f32_to_bf16_bits(a)


def zero_blocks(rng: np.random.Generator, bits: np.ndarray, frac=0.01, block=16) -> np.ndarray:
    """Zero a fraction of the 16-element blocks along the last dim (in place)."""
    rows, cols = bits.shape
    nblk = rows * (cols // block)
    pick = rng.choice(nblk, size=int(round(frac * nblk)), replace=False)
    v = bits.reshape(rows, cols // block, block)
    v[pick // (cols // block), pick % (cols // block), :] = 0
    return bits


# --------------------------------------------------------------- recipes
def single_linear(M=16, N=512, K=256, seed=0):
    """Single NVFP4 linear: A [M x K] ~N(0,1), W [N x K] ~N(0, 0.02), one
    stream (W drawn after A)."""
    rng = np.random.default_rng(seed)
    a = normal(rng, (M, K))
    w = normal(rng, (N, K), std=0.02)
    return a, w


def norm_weight(seed: int, n=H) -> np.ndarray:
    """RMSNorm weight ~ 1 + N(0, 0.05)."""
    return normal(np.random.default_rng(seed), (n,), mean=1.0, std=0.05)


def weight(seed: int, rows: int, cols: int, std=0.02, zero_block_frac=0.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    w = normal(rng, (rows, cols), std=std)
    if zero_block_frac:
        zero_blocks(rng, w, zero_block_frac)
    return w


def mlp_weights(layer: int = 0, h=H, i=I, zero_block_frac=0.0):
    """Gate [I x H], up [I x H], down [H x I] and the MLP norm weight for a
    layer; layer 0 uses seeds 11, 12, 13 (norm 17), layer l>0 uses 100+10l+j."""
    base = (lambda j: 10 + j) if layer == 0 else (lambda j: 100 + 10 * layer + j)
    return dict(
        w_gate=weight(base(1), i, h, zero_block_frac=zero_block_frac),
        w_up=weight(base(2), i, h, zero_block_frac=zero_block_frac),
        w_down=weight(base(3), h, i, zero_block_frac=zero_block_frac),
        mlp_norm=norm_weight(base(7), h),
    )


def attn_weights(layer: int = 0, h=H, qkv=QKV):
    """QKV [7168 x H], O [H x H] and the attention norm weight."""
    base = (lambda j: 10 + j) if layer == 0 else (lambda j: 100 + 10 * layer + j)
    return dict(
        w_qkv=weight(base(4), qkv, h),
        w_o=weight(base(5), h, h),
        attn_norm=norm_weight(base(6), h),
    )


def activations(T: int, seed: int, h=H, outliers=False) -> np.ndarray:
    rng = np.random.default_rng(seed)
    if outliers:
        return student_t_outliers(rng, (T, h))
    return normal(rng, (T, h))


def rope_tables(positions: int, rope_dim: int, theta: float = 10000.0):
    """cos and sin tables, float32 [positions, rope_dim/2], of the usual
    rotary angles p * theta^(-2i/rope_dim) (computed in float64, rounded
    once): inputs of the rotary embedding, not part of the NVFP4 path."""
    i = np.arange(rope_dim // 2, dtype=np.float64)
    ang = np.arange(positions, dtype=np.float64)[:, None] * theta ** (-2.0 * i / rope_dim)[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
