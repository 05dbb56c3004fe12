"""fp64 reference of rotary position embeddings (RoPE) on the mixer's q and k.

TEST INFRASTRUCTURE ONLY: the test suite and the benchmark's CPU baseline are its only
callers; it shares nothing with the CUDA library.  The pages embed the token mixer in a
Llama-style decoder with rotary position embeddings ("Interdomain Attention: Beyond
Token-Level Key-Value Memory", German technical summary, "Skalierbare Implementierung",
"Architektur"); as in that decoder the rotation is applied to the query and key rows
before the mixer.  Reading (the pages give no formula): channel pairs (2i, 2i + 1) of a
row at position p are rotated by the angle p * base^(-2i / R), base 10000 by default,
as the original rotary embedding of Llama does.
"""
from __future__ import annotations

import numpy as np


def angles(positions: np.ndarray, R: int, base: float = 10000.0) -> np.ndarray:
    """[P, R/2] rotation angles p * base^(-2i/R)."""
    inv = base ** (-np.arange(0, R, 2, dtype=np.float64) / R)
    return np.asarray(positions, np.float64)[:, None] * inv[None, :]


def rope(x: np.ndarray, pos0: int = 0, base: float = 10000.0) -> np.ndarray:
    """x [B, N, H, R] (read as float64), positions pos0 .. pos0 + N - 1 along axis 1."""
    x = np.asarray(x, np.float64)
    N, R = x.shape[1], x.shape[3]
    th = angles(np.arange(pos0, pos0 + N), R, base)[None, :, None, :]
    c, s = np.cos(th), np.sin(th)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out
