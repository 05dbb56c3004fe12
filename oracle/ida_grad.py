"""fp64 reference for the gradients of the Interdomain Attention token mixer.

TEST INFRASTRUCTURE ONLY: the test suite is its only caller.  It shares nothing
with the CUDA library (the seeded input generator aside) and nothing with the C
oracle: it is a second, independent restatement of the forward pass, written
with plain PyTorch CPU ops in float64 / complex128, whose gradients come from
autograd.  It is pinned by agreement with the C oracle's forward and by
finite differences (torch.autograd.gradcheck).  The library's backward pass
(ida_backward) is checked against it.

The forward follows "Interdomain Attention: Beyond Token-Level Key-Value Memory"
(German technical summary, "Skalierbare Implementierung"; the ratio readout
from its "Theoretische Herleitung"), step by step and in the same readings as
the C oracle:
  s    = causal depthwise conv of q and k (tap W-1 on the current position)
  xi   = SiLU(s) / (||SiLU(s)||^2 + eps_f)            (l_2 reading: / (||.|| + eps_f))
  kt   = RMSNorm(xi(k)) w_k + b_k,   vt = RMSNorm(v) w_v + b_v
  X_t  = lambda X_{t-1} + B [kt_t ; vt_t],  eta_t = lambda eta_{t-1} + B
  a_t  = xi(q_t) . U_t,   o_t = Re sum_m a_t[m] Gamma_t[m]   (eta readout: / Re sum_m a_t[m] eta_t[m])
"""
from __future__ import annotations

import torch

EPS_FEAT = 1e-6
EPS_RMS = 1e-6
READOUT_ETA = 1
FEAT_L2 = 2


def _conv(x: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
    """x [N, C], w [C, W]: s[t, c] = sum_j w[c, j] x[t - W + 1 + j, c], zeros before t = 0."""
    N, C = x.shape
    W = w.shape[1]
    xp = torch.cat([torch.zeros(W - 1, C, dtype=x.dtype), x], 0)
    return sum(w[:, j] * xp[j:j + N] for j in range(W))


def _feature(s: torch.Tensor, l2: bool) -> torch.Tensor:
    f = torch.nn.functional.silu(s)
    sq = (f * f).sum(1, keepdim=True)
    return f / ((torch.sqrt(sq) if l2 else sq) + EPS_FEAT)


def _rmsnorm(x: torch.Tensor, w: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    return x / torch.sqrt((x * x).mean(1, keepdim=True) + EPS_RMS) * w + b


def unit_forward(q, k, v, wq, wk, nw, bs, lam_ri, b_ri, flags: int = 0) -> torch.Tensor:
    """One (b,h) unit, float64 tensors: q, k [N, R], v [N, d], wq/wk [R, W], nw/bs [R+d],
    lam_ri/b_ri [M, 2].  Returns o [N, d]."""
    R = q.shape[1]
    l2 = bool(flags & FEAT_L2)
    xq = _feature(_conv(q, wq), l2)
    kt = _rmsnorm(_feature(_conv(k, wk), l2), nw[:R], bs[:R])
    vt = _rmsnorm(v, nw[R:], bs[R:])
    lam = torch.complex(lam_ri[:, 0], lam_ri[:, 1])
    Bv = torch.complex(b_ri[:, 0], b_ri[:, 1])
    M = lam.shape[0]
    U = torch.zeros(M, R, dtype=torch.complex128)
    G = torch.zeros(M, vt.shape[1], dtype=torch.complex128)
    eta = torch.zeros(M, dtype=torch.complex128)
    outs = []
    for t in range(q.shape[0]):
        U = lam[:, None] * U + Bv[:, None] * kt[t][None, :].to(torch.complex128)
        G = lam[:, None] * G + Bv[:, None] * vt[t][None, :].to(torch.complex128)
        eta = lam * eta + Bv
        a = U @ xq[t].to(torch.complex128)  # [M]
        o = (a[:, None] * G).sum(0).real
        if flags & READOUT_ETA:
            o = o / (a * eta).sum().real
        outs.append(o)
    return torch.stack(outs, 0)


def forward(q, k, v, params: dict, flags: int = 0) -> torch.Tensor:
    """[B, N, H, *] inputs (any float dtype; upcast to float64), the library's parameter
    layout (conv_w [2,H,R,W], norm_w/bias [H,R+d], lambda/Bvec [H,M,2]).  Returns out
    [B, N, H, d] float64, differentiable with respect to every float64 leaf passed in."""
    B, N, H, _ = q.shape
    outs = torch.stack([torch.stack([
        unit_forward(q[b, :, h], k[b, :, h], v[b, :, h], params["conv_w"][0, h], params["conv_w"][1, h],
                     params["norm_w"][h], params["bias"][h], params["lambda"][h], params["Bvec"][h], flags)
        for h in range(H)], 1) for b in range(B)], 0)
    return outs


def gradients(q, k, v, params: dict, grad_out: torch.Tensor, flags: int = 0) -> dict:
    """d<grad_out, out> with respect to q, k, v and every parameter, all float64."""
    leaves = {"q": q, "k": k, "v": v}
    leaves.update({n: params[n] for n in ("conv_w", "norm_w", "bias", "lambda", "Bvec")})
    leaves = {n: t.detach().to(torch.float64).requires_grad_(True) for n, t in leaves.items()}
    out = forward(leaves["q"], leaves["k"], leaves["v"], leaves, flags)
    g = torch.autograd.grad(out, list(leaves.values()), grad_outputs=grad_out.to(torch.float64))
    return dict(zip(leaves.keys(), g))
