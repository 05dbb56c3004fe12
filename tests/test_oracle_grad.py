"""Pins of the fp64 gradient reference (oracle/ida_grad.py): its forward is a second,
independent restatement and must agree with the C oracle; its gradients must agree
with finite differences of that forward."""
import numpy as np
import pytest
import torch

from oracle import ida_grad as og
from oracle import ida_oracle as orc
from linear_token_mixer_sc_gb300 import inputs


def _problem(B, N, H, R, d, M, W, seed, complex_b=True):
    p = inputs.make_params(H, R, d, M, W, seed)
    if complex_b:  # exercise the phase of B as well
        rng = np.random.default_rng(seed)
        p["Bvec"] = np.ascontiguousarray(rng.standard_normal((H, M, 2)) * 0.7, dtype=np.float32)
    q, k, v = inputs.make_qkv(B, N, H, R, d, "f32", seed)
    return q, k, v, p


def _t(p):
    return {n: torch.from_numpy(np.asarray(p[n], dtype=np.float64)) for n in
            ("conv_w", "norm_w", "bias", "lambda", "Bvec")}


@pytest.mark.parametrize("flags", [0, og.READOUT_ETA, og.FEAT_L2, og.READOUT_ETA | og.FEAT_L2])
def test_forward_matches_the_c_oracle(flags):
    q, k, v, p = _problem(2, 13, 2, 8, 6, 5, 4, seed=51)
    got = og.forward(q.double(), k.double(), v.double(), _t(p), flags).numpy()
    ref = orc.forward(q, k, v, p, flags=flags)["out"]
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("flags", [0, og.FEAT_L2, og.READOUT_ETA])
def test_gradients_match_finite_differences(flags):
    q, k, v, p = _problem(1, 5, 1, 4, 3, 2, 3, seed=52)
    pt = _t(p)
    names = ("q", "k", "v", "conv_w", "norm_w", "bias", "lambda", "Bvec")
    leaves = [q.double(), k.double(), v.double()] + [pt[n] for n in names[3:]]
    leaves = [x.clone().requires_grad_(True) for x in leaves]

    def fn(*xs):
        params = dict(zip(names[3:], xs[3:]))
        return og.forward(xs[0], xs[1], xs[2], params, flags)

    assert torch.autograd.gradcheck(fn, leaves, eps=1e-6, atol=1e-6, rtol=1e-4)


def test_gradients_entry_returns_every_input():
    q, k, v, p = _problem(1, 7, 2, 8, 6, 3, 4, seed=53)
    go = torch.randn(1, 7, 2, 6, dtype=torch.float64)
    g = og.gradients(q, k, v, _t(p), go)
    assert set(g) == {"q", "k", "v", "conv_w", "norm_w", "bias", "lambda", "Bvec"}
    assert g["q"].shape == q.shape and g["lambda"].shape == (2, 3, 2)
    # gradients are linear in the output gradient: a zero one gives zero gradients
    z = og.gradients(q, k, v, _t(p), torch.zeros_like(go))
    assert all(float(t.abs().max()) == 0.0 for t in z.values())
