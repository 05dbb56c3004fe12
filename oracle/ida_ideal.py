"""fp64 reference of the ideal Interdomain Attention derivation (random Fourier features).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU
baseline are its only callers.  It shares nothing with the CUDA library (the seeded
input generator aside) and nothing with the C oracle.  Plain NumPy in float64 /
complex128, following the translated paper text of "Interdomain Attention: Beyond
Token-Level Key-Value Memory" in its order:

  Eq. 1  attention as Nadaraya-Watson kernel regression,
         o_i = sum_n K(q_i, k_n) v_n / sum_n K(q_i, k_n);
  Eq. 3  a finite feature map, K(q, k) ~ xi(q)^T xi(k);
  Eq. 4  the resulting ratio, o_i ~ sum_n xi(q_i)^T xi(k_n) v_n / sum_n xi(q_i)^T xi(k_n);
  Eqs. 5-6  random Fourier features for a stationary kernel (Bochner):
         K(x, x') = E_omega[xi_omega(x)^T xi_omega(x')], xi_omega(x) = [cos(omega^T x), sin(omega^T x)];
  Fig. 1b  the interdomain layer: keys and values compressed by the SSM recurrence into
         U (M x R, key features), Gamma (M x d, values) and eta (M x 1, normaliser), read
         out as F_q U^T Gamma / (F_q U^T eta).

Readings where the pages stop (the text ends inside section 3.1, before the HiPPO
projection is specified): D frequencies omega_i (rows of a [D, R_in] matrix, drawn by the
caller, so they are inputs) give xi(x) = D^-1/2 [cos(Omega x); sin(Omega x)] in R^(2D),
whose inner products average the D frequencies; the causal form sums over n <= i; the
recurrence is the scalable layer's (X_t = lambda X_{t-1} + B [xi(k_t); v_t], eta_t =
lambda eta_{t-1} + B, no conjugation, real part taken last), applied directly to the
Fourier features with no conv and no normalisation, which the derivation does not have.
"""
from __future__ import annotations

import numpy as np


def rff(x: np.ndarray, omega: np.ndarray) -> np.ndarray:
    """Eqs. 5-6 with D frequencies: x [..., R_in], omega [D, R_in] -> [..., 2D]
    = D^-1/2 [cos(omega_i . x), sin(omega_i . x)]_i."""
    th = np.asarray(x, np.float64) @ np.asarray(omega, np.float64).T
    D = omega.shape[0]
    return np.concatenate([np.cos(th), np.sin(th)], axis=-1) / np.sqrt(D)


def gaussian_kernel(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """The stationary kernel whose spectral density is N(0, I): exp(-||x - y||^2 / 2)."""
    d2 = ((np.asarray(x, np.float64)[:, None, :] - np.asarray(y, np.float64)[None, :, :]) ** 2).sum(-1)
    return np.exp(-0.5 * d2)


def kernel_regression(q: np.ndarray, k: np.ndarray, v: np.ndarray, K: np.ndarray | None = None) -> np.ndarray:
    """Eq. 1, causal: o_i = sum_{n <= i} K(q_i, k_n) v_n / sum_{n <= i} K(q_i, k_n), one
    sequence (q, k [N, R_in], v [N, d]); K [N, N] given, or the Gaussian kernel."""
    if K is None:
        K = gaussian_kernel(q, k)
    N = q.shape[0]
    out = np.zeros((N, v.shape[1]))
    for i in range(N):
        w = K[i, : i + 1]
        out[i] = (w @ v[: i + 1]) / w.sum()
    return out


def linear_attention(fq: np.ndarray, fk: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Eq. 4, causal, by its definition: o_i = sum_{n <= i} (fq_i . fk_n) v_n /
    sum_{n <= i} (fq_i . fk_n), for feature rows fq, fk [N, F] and values v [N, d]."""
    N = fq.shape[0]
    out = np.zeros((N, v.shape[1]))
    for i in range(N):
        w = fk[: i + 1] @ fq[i]
        out[i] = (w @ v[: i + 1]) / w.sum()
    return out


def ideal_unit(q, k, v, omega, lam, B, final_state: bool = False):
    """The interdomain layer of Fig. 1b on Fourier features, one (b, h) unit, step by step:
    q, k [N, R_in], v [N, d], omega [D, R_in], lam and B [M] complex.  Returns o [N, d]
    (and the state [U | Gamma], eta after the last position)."""
    fq, fk = rff(q, omega), rff(k, omega)
    v = np.asarray(v, np.float64)
    M = lam.shape[0]
    U = np.zeros((M, fk.shape[1]), np.complex128)
    G = np.zeros((M, v.shape[1]), np.complex128)
    eta = np.zeros(M, np.complex128)
    out = np.zeros((q.shape[0], v.shape[1]))
    for t in range(q.shape[0]):
        U = lam[:, None] * U + B[:, None] * fk[t][None, :]
        G = lam[:, None] * G + B[:, None] * v[t][None, :]
        eta = lam * eta + B
        a = U @ fq[t]
        out[t] = (a[:, None] * G).sum(0).real / (a * eta).sum().real
    if final_state:
        return out, (U, G, eta)
    return out


def ideal_forward(q, k, v, omega, lam_ri, b_ri):
    """[B, N, H, *] inputs (any float dtype: read as float64), omega [H, D, R_in],
    lam_ri / b_ri [H, M, 2] (re, im).  Returns out [B, N, H, d] float64."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    Bn, N, H, _ = q.shape
    out = np.zeros((Bn, N, H, v.shape[3]))
    lam = lam_ri[..., 0] + 1j * lam_ri[..., 1]
    Bc = b_ri[..., 0] + 1j * b_ri[..., 1]
    for b in range(Bn):
        for h in range(H):
            out[b, :, h] = ideal_unit(q[b, :, h], k[b, :, h], v[b, :, h], omega[h], lam[h], Bc[h])
    return out
