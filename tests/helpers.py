"""Shared test utilities: error metrics and small problem builders."""
from __future__ import annotations

import numpy as np
import torch

from linear_token_mixer_sc_gb300 import inputs

# Tolerances stated for the mixer: fp32 inputs rel-L2 <= 1e-5 and max-abs
# <= 1e-4; bf16 inputs rel-L2 <= 3e-3.  The max-abs bar is applied to the
# error beyond the rounding of the exact result to the fp32 output format
# (``max_abs_beyond_rounding``): the workloads' outputs reach |o| ~ 1e4,
# where half an fp32 ulp is already 4.9e-4, so the oracle's own fp64 value
# stored as fp32 would miss a plain 1e-4 bar.
F32_REL_L2, F32_MAX_ABS = 1e-5, 1e-4
BF16_REL_L2 = 3e-3


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def max_abs(got, ref) -> float:
    return float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))))


def max_abs_beyond_rounding(got, ref) -> float:
    """max_i |got_i - ref_i| - ulp32(ref_i) / 2: the absolute error left after
    the unavoidable rounding of the exact value ref_i to an fp32 output."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    half_ulp = 0.5 * np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    return float(np.max(np.abs(got - ref) - half_ulp))


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def problem(B, N, H, R, d, M, W, dtype, seed):
    p = inputs.make_params(H, R, d, M, W, seed)
    q, k, v = inputs.make_qkv(B, N, H, R, d, dtype, seed)
    return q, k, v, p


def unpadded_state(st: np.ndarray, d: int, R: int, M: int, W: int) -> np.ndarray:
    """Drop the library's trailing alignment padding from [..., S] states."""
    n = 2 * M * (R + d) + 2 * M + 2 * (W - 1) * R
    return st[..., :n]


def head_params(p: dict, h: int) -> dict:
    """The parameters of head h alone, as a one-head parameter set."""
    return {"conv_w": p["conv_w"][:, h:h + 1], "norm_w": p["norm_w"][h:h + 1],
            "bias": p["bias"][h:h + 1], "lambda": p["lambda"][h:h + 1], "Bvec": p["Bvec"][h:h + 1]}
