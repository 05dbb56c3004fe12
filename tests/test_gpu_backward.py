"""GPU parity of ida_backward (gradients of the prefill) against the fp64 autograd
reference ``oracle/ida_grad.py`` (itself pinned to the C oracle's forward and to
finite differences).  Every gradient tensor is compared element by element on
the same seeded inputs: q, k, v and all five parameters, for both readouts and
both feature-map readings, with ragged chunk tails, N = 1, W < 4, d != R and odd M.
Tolerances: the forward's, rel-L2 <= 1e-5 for fp32 inputs (the kernels compute in
fp64) and <= 3e-3 for bf16 inputs (fp32 arithmetic, bf16 dq, dk, dv).
"""
import numpy as np
import pytest
import torch

from linear_token_mixer_sc_gb300 import binding, build, inputs
from oracle import ida_grad as og
from tests.helpers import BF16_REL_L2, F32_REL_L2, rel_l2

pytestmark = pytest.mark.gpu

ETA, L2 = binding.IDA_READOUT_ETA, binding.IDA_FEAT_L2
NAMES = ("q", "k", "v", "conv_w", "norm_w", "bias", "lambda", "Bvec")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _case(B, N, H, R, d, M, W, dt, seed, complex_b=True):
    p = inputs.make_params(H, R, d, M, W, seed)
    if complex_b:  # a complex B with modulus around 1 exercises the phase of B as well
        rng = np.random.default_rng(seed)
        phase = rng.uniform(-np.pi, np.pi, (H, M))
        p["Bvec"] = np.ascontiguousarray(np.stack([np.cos(phase), np.sin(phase)], -1), dtype=np.float32)
    q, k, v = inputs.make_qkv(B, N, H, R, d, dt, seed)
    g = torch.Generator().manual_seed(seed)
    dout = torch.randn(B, N, H, d, generator=g).to(inputs.torch_dtype(dt))
    return q, k, v, p, dout


def _gpu(q, k, v, p, dout, flags):
    dev = torch.device("cuda")
    pd = binding.params_to_device(p)
    g = binding.ida_backward(q.to(dev), k.to(dev), v.to(dev), pd, dout.to(dev), flags=flags)
    torch.cuda.synchronize()
    assert binding.ida_device_error() == 0
    return {n: t.float().cpu().double().numpy() for n, t in g.items()}


def _ref(q, k, v, p, dout, flags):
    pt = {n: torch.from_numpy(np.asarray(p[n], dtype=np.float64)) for n in NAMES[3:]}
    g = og.gradients(q.double(), k.double(), v.double(), pt, dout.double(), flags)
    return {n: t.numpy() for n, t in g.items()}


# (B, N, H, R, d, M, W, dtype, flags)
CASES = [
    (1, 70, 2, 32, 32, 16, 4, "f32", 0),          # a ragged second chunk of 64
    (2, 37, 1, 16, 24, 5, 3, "f32", ETA),         # d != R, odd M, W = 3, eta readout, two batch rows
    (1, 130, 1, 32, 16, 8, 2, "f32", L2),         # three chunks, the l_2 feature map
    (1, 1, 2, 8, 8, 3, 4, "f32", 0),              # one position
    (2, 50, 2, 16, 16, 7, 1, "f32", ETA | L2),    # W = 1 (no conv history)
    (1, 80, 1, 64, 64, 64, 4, "f32", ETA),        # modes split over two CTAs, eta readout
    (2, 150, 2, 64, 64, 64, 4, "bf16", 0),        # the tensor-core forward's shape class (two mode slices)
    (1, 90, 2, 64, 32, 16, 4, "bf16", L2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}N{}H{}R{}d{}M{}W{}{}f{}".format(*c))
def test_backward_matches_autograd_reference(case):
    B, N, H, R, d, M, W, dt, flags = case
    q, k, v, p, dout = _case(B, N, H, R, d, M, W, dt, seed=700 + N)
    got = _gpu(q, k, v, p, dout, flags)
    ref = _ref(q, k, v, p, dout, flags)
    tol = F32_REL_L2 if dt == "f32" else BF16_REL_L2
    errs = {n: rel_l2(got[n], ref[n]) for n in NAMES}
    assert all(e <= tol for e in errs.values()), errs
    for n in NAMES:
        assert got[n].shape == ref[n].shape, n


def test_backward_is_deterministic():
    q, k, v, p, dout = _case(2, 100, 2, 32, 32, 16, 4, "bf16", seed=11)
    dev = torch.device("cuda")
    pd = binding.params_to_device(p)
    args = (q.to(dev), k.to(dev), v.to(dev), pd, dout.to(dev))
    g1 = binding.ida_backward(*args)
    g2 = binding.ida_backward(*args)
    torch.cuda.synchronize()
    for n in NAMES:
        assert torch.equal(g1[n], g2[n]), n


def test_backward_of_zero_output_gradient_is_zero():
    q, k, v, p, dout = _case(1, 40, 2, 32, 32, 8, 4, "f32", seed=12)
    got = _gpu(q, k, v, p, torch.zeros_like(dout), 0)
    for n in NAMES:
        assert np.count_nonzero(got[n]) == 0, n


def test_backward_zero_length_gives_zero_parameter_gradients():
    B, H, R, d, M, W = 1, 2, 16, 16, 4, 4
    p = inputs.make_params(H, R, d, M, W, 3)
    e = torch.empty((B, 0, H, R), dtype=torch.float32, device="cuda")
    ev = torch.empty((B, 0, H, d), dtype=torch.float32, device="cuda")
    g = binding.ida_backward(e, e.clone(), ev, binding.params_to_device(p), ev.clone())
    torch.cuda.synchronize()
    for n in NAMES[3:]:
        assert torch.count_nonzero(g[n]).item() == 0, n


def test_backward_full_125m_shape_sampled_head():
    """The benchmark's backward workload as it launches it (B=8, H=12, N=2048, R=d=64, M=64,
    bf16, with a caller workspace: two mode slices per unit, 192 CTAs), checked against the
    autograd reference on every batch row of one head: dq, dk, dv of those 8 units and the
    head's parameter gradients (sums over the batch rows), each over all positions."""
    from linear_token_mixer_sc_gb300 import configs
    w = configs.PREFILL_125M
    p = inputs.make_params(w.H, w.R, w.d, w.M, w.W, w.seed)
    q, k, v = inputs.make_qkv(w.B, w.N, w.H, w.R, w.d, w.dtype, w.seed)
    g = torch.Generator().manual_seed(w.seed + 1000)
    dout = torch.randn(w.B, w.N, w.H, w.d, generator=g).to(q.dtype)
    dev = torch.device("cuda")
    nb = binding.ida_backward_workspace_bytes(w.B, w.H, w.N, w.d, w.R, w.M, binding.IDA_BF16, w.W, 0)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    got = binding.ida_backward(q.to(dev), k.to(dev), v.to(dev), binding.params_to_device(p), dout.to(dev),
                               workspace=ws)
    torch.cuda.synchronize()
    assert binding.ida_device_error() == 0
    h = 5
    hs = slice(h, h + 1)
    ps = {"conv_w": p["conv_w"][:, hs], "norm_w": p["norm_w"][hs], "bias": p["bias"][hs],
          "lambda": p["lambda"][hs], "Bvec": p["Bvec"][hs]}
    ref = _ref(q[:, :, hs], k[:, :, hs], v[:, :, hs], ps, dout[:, :, hs], 0)
    gh = {n: got[n].float().cpu().double().numpy() for n in NAMES}
    sel = {"q": gh["q"][:, :, hs], "k": gh["k"][:, :, hs], "v": gh["v"][:, :, hs],
           "conv_w": gh["conv_w"][:, hs], "norm_w": gh["norm_w"][hs], "bias": gh["bias"][hs],
           "lambda": gh["lambda"][hs], "Bvec": gh["Bvec"][hs]}
    errs = {n: rel_l2(sel[n], ref[n]) for n in NAMES}
    assert all(e <= BF16_REL_L2 for e in errs.values()), errs
