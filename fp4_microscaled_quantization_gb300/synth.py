"""Seeded synthetic operands shaped like the pages' Llama-3.1-8B-class workloads.

This module only draws random numbers and rounds them to bf16; it holds none
of the quantizer's arithmetic.  Both the CUDA path's tests/benchmark and the
CPU oracle's tests take their inputs from here.

Every tensor is drawn with ``numpy.random.Generator(PCG64(seed))`` in fp32 and
rounded to bf16 with round-to-nearest-even by torch.  Tensors are returned as
``uint16`` arrays of bf16 bit patterns (row-major); ``as_torch`` views them as
``torch.bfloat16``.

Workloads (hidden size 4096, FFN size 14336, 8192/16384 tokens):
  tiny      X 256 x 512,   N(0,1), 1% of positions (seeded) x 50
  act       X 8192 x 4096, N(0,1), 8 seeded channels (whole columns) x 30
  grad      dY 8192 x 14336, Student-t(3) * 1e-3
  weight    W 14336 x 4096, N(0, 0.02^2)
  layer     X 16384 x 4096 (act distribution), W 4096 x 4096 (weight
            distribution), dY 16384 x 4096 (grad distribution)
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch

SEED_BASE = 1000


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (RNE, via torch) and return the uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def as_torch(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def sha256(bits: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(bits).tobytes()).hexdigest()


# ------------------------------------------------------------ distributions
def normal(rows: int, cols: int, seed: int, std: float = 1.0) -> np.ndarray:
    g = _rng(seed)
    x = g.standard_normal((rows, cols), dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return to_bf16_bits(x)


def normal_point_outliers(rows: int, cols: int, seed: int, frac: float = 0.01, mult: float = 50.0) -> np.ndarray:
    """N(0,1) with round(frac * rows * cols) positions, drawn without replacement, scaled by mult."""
    g = _rng(seed)
    x = g.standard_normal((rows, cols), dtype=np.float32)
    n_out = int(round(frac * rows * cols))
    pos = g.choice(rows * cols, size=n_out, replace=False)
    x.reshape(-1)[pos] *= np.float32(mult)
    return to_bf16_bits(x)


def normal_channel_outliers(rows: int, cols: int, seed: int, n_channels: int = 8, mult: float = 30.0) -> np.ndarray:
    """N(0,1) with n_channels seeded whole columns scaled by mult."""
    g = _rng(seed)
    x = g.standard_normal((rows, cols), dtype=np.float32)
    ch = g.choice(cols, size=min(n_channels, cols), replace=False)
    x[:, ch] *= np.float32(mult)
    return to_bf16_bits(x)


def student_t(rows: int, cols: int, seed: int, df: float = 3.0, scale: float = 1e-3) -> np.ndarray:
    g = _rng(seed)
    x = np.empty((rows, cols), dtype=np.float32)
    step = max(1, (1 << 24) // max(cols, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x[r0:r1] = (g.standard_t(df, size=(r1 - r0, cols)) * scale).astype(np.float32)
    return to_bf16_bits(x)


def special_values(rows: int, cols: int, seed: int) -> np.ndarray:
    """Edge-case mix: zeros (both signs), tiny and subnormal bf16 values, exact
    grid midpoints at several binades, constant blocks and large magnitudes."""
    g = _rng(seed)
    x = g.standard_normal((rows, cols), dtype=np.float32)
    flat = x.reshape(-1)
    n = flat.size
    pick = lambda k: g.choice(n, size=min(k, n), replace=False)
    flat[pick(n // 16)] = 0.0
    flat[pick(n // 32)] = -0.0
    flat[pick(n // 32)] = np.float32(1e-39) * g.standard_normal(min(n // 32, n)).astype(np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.125, 0.375, 0.625, 0.875, 1.125, 1.375, 1.625],
                    dtype=np.float32)
    idx = pick(n // 8)
    flat[idx] = mids[g.integers(0, mids.size, idx.size)] * np.float32(2.0) ** g.integers(-3, 4, idx.size).astype(np.float32)
    flat[idx] *= np.where(g.random(idx.size) < 0.5, -1.0, 1.0).astype(np.float32)
    flat[pick(n // 64)] *= np.float32(1e30)
    xr = x.reshape(rows, cols)
    if rows >= 32 and cols >= 32:
        xr[0:32, 0:32] = 0.0          # an all-zero block in both orientations
        xr[0:32, 32:64] = 3.0         # a constant block
    return to_bf16_bits(xr)


# ------------------------------------------------------------ workloads
def tiny_x():
    return normal_point_outliers(256, 512, SEED_BASE + 1, 0.01, 50.0)


def act_x(rows: int = 8192, cols: int = 4096, seed: int = SEED_BASE + 2):
    return normal_channel_outliers(rows, cols, seed, 8, 30.0)


def grad_dy(rows: int = 8192, cols: int = 14336, seed: int = SEED_BASE + 3):
    return student_t(rows, cols, seed, 3.0, 1e-3)


def weight_w(rows: int = 14336, cols: int = 4096, seed: int = SEED_BASE + 4):
    return normal(rows, cols, seed, 0.02)


def layer(tokens: int = 16384, d_in: int = 4096, d_out: int = 4096, seed: int = SEED_BASE + 5):
    """One linear layer's operands: X [tokens, d_in], W [d_out, d_in], dY [tokens, d_out]."""
    X = act_x(tokens, d_in, seed * 10 + 1)
    W = weight_w(d_out, d_in, seed * 10 + 2)
    dY = grad_dy(tokens, d_out, seed * 10 + 3)
    return X, W, dY


def grid_valued(rows: int, cols: int, seed: int, grid: int = 0) -> np.ndarray:
    """Entries drawn uniformly from the signed levels of a 4-bit grid (0: E2M1
    {0, .5, 1, 1.5, 2, 3, 4, 6}; 1: E1M2 {k/4}), with one seeded position of
    every 32-element row block set to a level of the grid's top binade (E2M1
    4 or 6; E1M2 1 .. 1.75).  Every block's power-of-two scale is then 1 and
    the values are their own quantization, so products of two such matrices
    are multiples of 1/4 (E2M1) or 1/16 (E1M2) whose sums stay exact in fp32
    for K <= 4096."""
    g = _rng(seed)
    levels = (np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float32) if grid == 0
              else np.arange(8, dtype=np.float32) / np.float32(4.0))
    top = levels[6:] if grid == 0 else levels[4:]
    x = levels[g.integers(0, 8, (rows, cols))]
    nb = cols // 32
    pos = g.integers(0, 32, (rows, nb)) + 32 * np.arange(nb)[None, :]
    x[np.arange(rows)[:, None], pos] = top[g.integers(0, top.size, (rows, nb))]
    x *= np.where(g.random((rows, cols)) < 0.5, -1.0, 1.0).astype(np.float32)
    return to_bf16_bits(x)
