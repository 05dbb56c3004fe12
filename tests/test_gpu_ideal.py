"""GPU parity of ida_forward_ideal (the ideal interdomain layer on random Fourier
features) against the fp64 oracle ``oracle/ida_ideal.py`` (pinned by Bochner's
identity, Eq. 4's recurrent form and closed forms of the layer).  Element by
element, rel-L2 <= 1e-5 for fp32 inputs and <= 3e-3 for bf16 inputs; odd shapes:
N = 1, ragged tiles, D not a multiple of 32, d != 2D, odd M, several heads."""
import numpy as np
import pytest
import torch

from linear_token_mixer_sc_gb300 import binding, build, inputs
from oracle import ida_ideal as ii
from tests.helpers import BF16_REL_L2, F32_REL_L2, rel_l2, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


# (B, N, H, R_in, D, d, M, dtype)
CASES = [
    (1, 1, 2, 16, 8, 8, 4, "f32"),
    (2, 37, 3, 32, 16, 32, 16, "f32"),
    (1, 70, 2, 24, 20, 16, 7, "f32"),
    (1, 200, 2, 64, 32, 64, 64, "f32"),
    (2, 130, 2, 64, 32, 64, 64, "bf16"),
    (1, 90, 4, 128, 64, 128, 64, "bf16"),
    # unit counts whose clusters fill one wave of two CTAs per SM with G = 5, 6, 7 on 152 SMs:
    # uneven mode ranges (13 x 4 + 12, 11 x 5 + 9, 10 x 6 + 4 modes)
    (4, 40, 13, 32, 16, 32, 64, "bf16"),
    (2, 30, 24, 32, 16, 32, 64, "bf16"),
    (5, 25, 8, 32, 16, 32, 64, "f32"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}N{}H{}Rin{}D{}d{}M{}{}".format(*c))
def test_ideal_layer_matches_oracle(case):
    B, N, H, Rin, D, d, M, dt = case
    seed = 900 + N
    p = inputs.make_params(H, Rin, d, M, 4, seed)
    q, k, v = inputs.make_qkv(B, N, H, Rin, d, dt, seed)
    om = inputs.make_omega(H, D, Rin, seed)
    dev = torch.device("cuda")
    out = binding.ida_forward_ideal(q.to(dev), k.to(dev), v.to(dev), torch.from_numpy(om).to(dev),
                                    binding.params_to_device(p))
    torch.cuda.synchronize()
    assert binding.ida_device_error() == 0
    ref = ii.ideal_forward(q.double().numpy(), k.double().numpy(), v.double().numpy(), om.astype(np.float64),
                           p["lambda"].astype(np.float64), p["Bvec"].astype(np.float64))
    err = rel_l2(to_np(out), ref)
    assert err <= (F32_REL_L2 if dt == "f32" else BF16_REL_L2), err


def test_ideal_layer_is_deterministic():
    B, N, H, Rin, D, d, M = 2, 100, 2, 32, 16, 32, 32
    p = inputs.make_params(H, Rin, d, M, 4, 5)
    q, k, v = inputs.make_qkv(B, N, H, Rin, d, "bf16", 5)
    om = torch.from_numpy(inputs.make_omega(H, D, Rin, 5)).cuda()
    pd = binding.params_to_device(p)
    o1 = binding.ida_forward_ideal(q.cuda(), k.cuda(), v.cuda(), om, pd)
    o2 = binding.ida_forward_ideal(q.cuda(), k.cuda(), v.cuda(), om, pd)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_ideal_layer_full_125m_shape_sampled_units():
    """The benchmark's ideal-layer workload as it launches it (B=8, H=12, N=2048, R_in = d = 64,
    D = 32 frequencies, M = 64, bf16: two-CTA clusters over 96 units), checked against the
    oracle on six (b,h) units spread over the batch and the heads, each over all positions."""
    from linear_token_mixer_sc_gb300 import configs
    w = configs.PREFILL_125M
    D = 32
    p = inputs.make_params(w.H, w.R, w.d, w.M, w.W, w.seed)
    q, k, v = inputs.make_qkv(w.B, w.N, w.H, w.R, w.d, w.dtype, w.seed)
    om = inputs.make_omega(w.H, D, w.R, w.seed)
    dev = torch.device("cuda")
    out = binding.ida_forward_ideal(q.to(dev), k.to(dev), v.to(dev), torch.from_numpy(om).to(dev),
                                    binding.params_to_device(p))
    torch.cuda.synchronize()
    assert binding.ida_device_error() == 0
    got = to_np(out)
    lam = p["lambda"][..., 0].astype(np.float64) + 1j * p["lambda"][..., 1].astype(np.float64)
    bc = p["Bvec"][..., 0].astype(np.float64) + 1j * p["Bvec"][..., 1].astype(np.float64)
    for b, h in [(0, 0), (1, 7), (3, 11), (4, 2), (6, 5), (7, 9)]:
        ref = ii.ideal_unit(q[b, :, h].double().numpy(), k[b, :, h].double().numpy(), v[b, :, h].double().numpy(),
                            om[h].astype(np.float64), lam[h], bc[h])
        err = rel_l2(got[b, :, h], ref)
        assert err <= BF16_REL_L2, (b, h, err)
