"""Seeded synthetic inputs shaped like the workloads of the packed formats.

This module only draws random bytes and numbers; it decodes nothing and
computes no product. Both the CUDA path and the oracle are fed from it, so
they always see identical bytes. All draws use NumPy's PCG64 generator.

Every recipe returns plain NumPy arrays (16-bit floats as uint16 bit
patterns) plus the metadata a caller needs to describe the weight:

* MLX affine: ``codes`` uint32 [..., n, k*bits/32] (codes uniform, so the
  words are uniform 32-bit values), ``scales`` and ``biases`` bf16
  [..., n, k/group_size].
* GGUF Q8_0: ``codes`` uint8 [..., n, k/32*34], each 34-byte block a
  little-endian float16 d = |N(0, sigma)| then 32 int8 quants uniform in
  [-127, 127].
* MXFP4: ``codes`` uint8 [..., n, k/2] uniform bytes, ``scales`` uint8
  [..., n, k/32] e8m0 bytes uniform in [lo, hi].
* MXFP4 in GGUF's blocks: ``codes`` uint8 [..., n, k/32*17], each 17-byte
  block an e8m0 byte uniform in [lo, hi] then 16 uniform bytes.
* GGUF Q4_K: ``codes`` uint8 [..., n, k/256*144], each 144-byte block a
  float16 d and dmin = |N(0, sigma)|, then 140 uniform bytes (the packed
  6-bit scales and mins, and the 4-bit quants).
* GGUF Q6_K: ``codes`` uint8 [..., n, k/256*210], each 210-byte block 192
  uniform bytes (quants), 16 int8 scales uniform in [-128, 127], then a
  float16 d = |N(0, sigma)|.
"""
from __future__ import annotations

import numpy as np
import torch

AFFINE, Q8_0, MXFP4, MXFP4_BLOCKS, Q4_K, Q6_K = "affine", "q8_0", "mxfp4", "mxfp4_blocks", "q4_k", "q6_k"


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> bfloat16 bit patterns (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_f16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).astype("<f2").view(np.uint16).copy()


def normal_bf16(g: np.random.Generator, shape, sigma=1.0, absolute=False, add=0.0):
    v = g.standard_normal(shape, dtype=np.float32) * np.float32(sigma)
    if absolute:
        v = np.abs(v)
    if add:
        v = v + np.float32(add)
    return to_bf16_bits(v)


def normal_f16(g: np.random.Generator, shape, sigma=1.0, absolute=False, add=0.0):
    """float16 bit patterns of N(0, sigma) draws (NumPy's conversion, round to nearest even)."""
    v = g.standard_normal(shape, dtype=np.float32) * np.float32(sigma)
    if absolute:
        v = np.abs(v)
    if add:
        v = v + np.float32(add)
    return v.astype(np.float16).view(np.uint16)


def affine_weight(g, n, k, bits=4, group_size=64, lead=(), scale_sigma=0.02, scale_add=0.0,
                  bias_sigma=0.02, scale_dtype="bf16"):
    """MLX affine weight [*lead, n, k]; scales and biases bf16 or f16."""
    assert (k * bits) % 32 == 0 and k % group_size == 0
    shape = tuple(lead) + (n,)
    codes = g.integers(0, 2**32, size=shape + (k * bits // 32,), dtype=np.uint64).astype(np.uint32)
    draw = normal_f16 if scale_dtype == "f16" else normal_bf16
    scales = draw(g, shape + (k // group_size,), scale_sigma, absolute=True, add=scale_add)
    biases = draw(g, shape + (k // group_size,), bias_sigma)
    return dict(format=AFFINE, shape=shape + (k,), bits=bits, group_size=group_size,
                scale_dtype=scale_dtype, codes=codes, scales=scales, biases=biases)


def q8_0_weight(g, n, k, lead=(), d_sigma=0.005):
    """GGUF Q8_0 weight [*lead, n, k]."""
    assert k % 32 == 0
    shape = tuple(lead) + (n,)
    nb = k // 32
    d = np.abs(g.standard_normal(shape + (nb,), dtype=np.float32) * np.float32(d_sigma))
    d_bytes = d.astype("<f2").view(np.uint8).reshape(shape + (nb, 2))
    q = g.integers(-127, 128, size=shape + (nb, 32), dtype=np.int64).astype(np.int8)
    blocks = np.concatenate([d_bytes, q.view(np.uint8)], axis=-1)
    return dict(format=Q8_0, shape=shape + (k,), bits=8, group_size=32, scale_dtype=None,
                codes=np.ascontiguousarray(blocks.reshape(shape + (nb * 34,))), scales=None,
                biases=None)


def mxfp4_weight(g, n, k, lead=(), scale_lo=118, scale_hi=126):
    """MXFP4 weight [*lead, n, k], scales apart."""
    assert k % 32 == 0
    shape = tuple(lead) + (n,)
    codes = g.integers(0, 256, size=shape + (k // 2,), dtype=np.int64).astype(np.uint8)
    scales = g.integers(scale_lo, scale_hi + 1, size=shape + (k // 32,), dtype=np.int64)
    return dict(format=MXFP4, shape=shape + (k,), bits=4, group_size=32, scale_dtype=None,
                codes=codes, scales=scales.astype(np.uint8), biases=None)


def mxfp4_blocks_weight(g, n, k, lead=(), scale_lo=118, scale_hi=126):
    """MXFP4 weight [*lead, n, k] in GGUF's 17-byte blocks."""
    assert k % 32 == 0
    shape = tuple(lead) + (n,)
    blocks = g.integers(0, 256, size=shape + (k // 32, 17), dtype=np.int64)
    blocks[..., 0] = g.integers(scale_lo, scale_hi + 1, size=shape + (k // 32,), dtype=np.int64)
    return dict(format=MXFP4_BLOCKS, shape=shape + (k,), bits=4, group_size=32, scale_dtype=None,
                codes=blocks.astype(np.uint8).reshape(shape + (k // 32 * 17,)), scales=None, biases=None)


def q4_k_weight(g, n, k, lead=(), d_sigma=0.002):
    """GGUF Q4_K weight [*lead, n, k] (k a multiple of 256)."""
    assert k % 256 == 0
    shape = tuple(lead) + (n,)
    nb = k // 256
    blocks = g.integers(0, 256, size=shape + (nb, 144), dtype=np.int64).astype(np.uint8)
    dd = np.abs(g.standard_normal(shape + (nb, 2), dtype=np.float32) * np.float32(d_sigma))
    blocks[..., 0:4] = dd.astype("<f2").view(np.uint8).reshape(shape + (nb, 4))
    return dict(format=Q4_K, shape=shape + (k,), bits=4, group_size=256, scale_dtype=None,
                codes=np.ascontiguousarray(blocks.reshape(shape + (nb * 144,))), scales=None, biases=None)


def q6_k_weight(g, n, k, lead=(), d_sigma=0.0005):
    """GGUF Q6_K weight [*lead, n, k] (k a multiple of 256)."""
    assert k % 256 == 0
    shape = tuple(lead) + (n,)
    nb = k // 256
    blocks = g.integers(0, 256, size=shape + (nb, 210), dtype=np.int64).astype(np.uint8)
    d = np.abs(g.standard_normal(shape + (nb,), dtype=np.float32) * np.float32(d_sigma))
    blocks[..., 208:210] = d.astype("<f2").view(np.uint8).reshape(shape + (nb, 2))
    return dict(format=Q6_K, shape=shape + (k,), bits=6, group_size=256, scale_dtype=None,
                codes=np.ascontiguousarray(blocks.reshape(shape + (nb * 210,))), scales=None, biases=None)


def activations(g, M, k, sigma=1.0):
    """x bf16 [M, k] ~ N(0, sigma^2)."""
    return normal_bf16(g, (M, k), sigma)


def expert_ids(g, T, topk, E):
    """int32 [T, topk]: distinct experts per row, uniform over E."""
    keys = g.random((T, E))
    return np.argsort(keys, axis=1)[:, :topk].astype(np.int32)


def uniform_ids(g, count, length):
    return g.integers(0, length, size=count, dtype=np.int64).astype(np.int32)


# ---------------------------------------------------------------- workloads
# Qwen3-0.6B-shaped projections (n, k): hidden 1024.
QWEN3_0_6B_LAYER = {
    "q_proj": (2048, 1024),
    "k_proj": (1024, 1024),
    "v_proj": (1024, 1024),
    "gate_proj": (3072, 1024),
    "up_proj": (3072, 1024),
    "down_proj": (1024, 3072),
}
QWEN3_0_6B_LM_HEAD = (151936, 1024)
QWEN3_0_6B_LAYERS = 28

Q8_0_SHAPES = [(4096, 4096), (14336, 4096), (4096, 14336)]


def small_affine_config(seed=0):
    """Affine 4-bit gs64, W 256x512: scales |N(0,.02)|+1e-3, biases N(0,.02), seed 0."""
    g = rng(seed)
    w = affine_weight(g, 256, 512, bits=4, group_size=64, scale_add=1e-3)
    xs = {M: activations(g, M, 512) for M in (1, 8)}
    return w, xs


def moe_config(T, seed=3, E=32, n=5760, k=2880, topk=4):
    """MXFP4 expert stack [E, n, k], scales in 118..126, ids [T, topk], x [T, k]."""
    g = rng(seed)
    w = mxfp4_weight(g, n, k, lead=(E,))
    ids = expert_ids(g, T, topk, E)
    x = activations(g, T, k)
    return w, ids, x
