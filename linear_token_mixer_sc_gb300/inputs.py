"""Seeded synthetic inputs for the Interdomain Attention token mixer.

This module is the one piece shared by the CUDA path and the CPU oracle's
tests.  It draws random numbers and nothing else: none of the mixer's
arithmetic lives here.

Recipe (the stand-in for the language-modelling workloads of "Interdomain
Attention: Beyond Token-Level Key-Value Memory", whose data and weights are
not available): q, k, v ~ N(0, 1); depthwise conv taps ~ N(0, 1/4) (variance,
i.e. std 1/2 = 1/sqrt(W) for W = 4); RMSNorm weights = 1; RMSNorm biases ~
N(0, 0.1) (variance); per head one step size Delta_h, log-uniform on
[1e-3, 1e-1], and modes lambda_{h,m} = exp(Delta_h (-1/2 + i pi m)) (S4D-Lin);
B_m = 1.  Parameters are drawn in float64 and stored as float32, the dtype
the library takes; both sides read the same float32 bytes.
"""
from __future__ import annotations

import math

import numpy as np
import torch

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _DT[name]


def make_params(H: int, R: int, d: int, M: int, W: int, seed: int,
                conv_var: float = 0.25, bias_var: float = 0.1,
                delta_range=(1e-3, 1e-1)) -> dict:
    """conv_w [2,H,R,W], norm_w/bias [H,R+d], lambda/Bvec [H,M,2] (float32)."""
    rng = np.random.default_rng([seed, 1])
    conv_w = rng.standard_normal((2, H, R, W)) * math.sqrt(conv_var)
    norm_w = np.ones((H, R + d))
    bias = rng.standard_normal((H, R + d)) * math.sqrt(bias_var)
    lo, hi = math.log(delta_range[0]), math.log(delta_range[1])
    delta = np.exp(rng.uniform(lo, hi, size=H))
    m = np.arange(M)
    lam = np.exp(delta[:, None] * (-0.5 + 1j * math.pi * m[None, :]))
    lam_ri = np.stack([lam.real, lam.imag], axis=-1)
    b_ri = np.zeros((H, M, 2))
    b_ri[..., 0] = 1.0
    f = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    return {"conv_w": f(conv_w), "norm_w": f(norm_w), "bias": f(bias),
            "lambda": f(lam_ri), "Bvec": f(b_ri), "delta": delta}


def make_qkv(B: int, N: int, H: int, R: int, d: int, dtype: str, seed: int,
             device: str | torch.device = "cpu"):
    """q, k [B,N,H,R] and v [B,N,H,d], N(0,1), cast to ``dtype``.

    On the CPU the draws come from NumPy's PCG64; on a CUDA device from
    torch's seeded device generator (used for inputs too large to draw on the
    host).  Either way the tensors returned are the inputs of record: the
    oracle reads exactly these bytes.
    """
    tdt = _DT[dtype]
    dev = torch.device(device)
    if dev.type == "cpu":
        rng = np.random.default_rng([seed, 0])
        out = []
        for shape in ((B, N, H, R), (B, N, H, R), (B, N, H, d)):
            a = rng.standard_normal(shape, dtype=np.float32)
            out.append(torch.from_numpy(a).to(tdt))
        return tuple(out)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    out = []
    for shape in ((B, N, H, R), (B, N, H, R), (B, N, H, d)):
        out.append(torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(tdt))
    return tuple(out)


def make_tokens(B: int, H: int, R: int, d: int, dtype: str, seed: int, step: int,
                device: str | torch.device = "cpu"):
    """One decode token per (b,h): q, k [B,H,R], v [B,H,d], N(0,1)."""
    tdt = _DT[dtype]
    dev = torch.device(device)
    if dev.type == "cpu":
        rng = np.random.default_rng([seed, 2, step])
        return tuple(torch.from_numpy(rng.standard_normal(s, dtype=np.float32)).to(tdt)
                     for s in ((B, H, R), (B, H, R), (B, H, d)))
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed) * 1000003 + int(step))
    return tuple(torch.randn(s, generator=g, device=dev, dtype=torch.float32).to(tdt)
                 for s in ((B, H, R), (B, H, R), (B, H, d)))


def make_omega(H: int, D: int, R_in: int, seed: int) -> np.ndarray:
    """Random Fourier frequencies for the ideal-derivation workload: [H, D, R_in] drawn
    from N(0, I / R_in) (the Gaussian kernel at the bandwidth of R_in-dimensional rows
    with unit-variance entries), stored as float32.  The draw is an input of the layer,
    read by the library and the oracle alike."""
    rng = np.random.default_rng([seed, 7])
    return np.ascontiguousarray(rng.standard_normal((H, D, R_in)) / math.sqrt(R_in), dtype=np.float32)
