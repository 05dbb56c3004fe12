"""GPU parity of ida_rope (rotary position embeddings on q and k, in place) against the
fp64 oracle ``oracle/ida_rope.py``, itself pinned by closed forms and invariants.

Bars, from the arithmetic: the angle is reduced modulo 2 pi exactly (a 64-bit fixed-point
phase), sin / cos and the rotation run in fp32, so an fp32 result is within a few fp32
ulps of the exact value (max-abs <= 2e-6 on unit-variance inputs, rel-L2 <= 1e-6); a bf16
result is the fp32 value rounded once to bf16, so each element is within half a bf16 ulp
(2^-8 |x|) plus that fp32 error of the exact value.
"""
import numpy as np
import pytest
import torch

from linear_token_mixer_sc_gb300 import binding, build, configs
from oracle import ida_rope as ro
from tests.helpers import rel_l2

pytestmark = pytest.mark.gpu

F32_ABS, F32_REL = 2e-6, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _x(B, N, H, R, seed, dt):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, N, H, R, generator=g)
    return x.to(torch.bfloat16) if dt == "bf16" else x


def _check(got, ref, x_in, dt):
    got = got.float().cpu().double().numpy()
    if dt == "f32":
        assert np.max(np.abs(got - ref)) <= F32_ABS
        assert rel_l2(got, ref) <= F32_REL
    else:
        bound = 2.0 ** -8 * np.abs(ref) + F32_ABS
        assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) - bound))


# (B, N, H, R, pos0, base, dtype)
CASES = [
    (2, 37, 3, 32, 0, 10000.0, "f32"),              # a ragged last tile of positions
    (1, 8, 1, 8, 0, 10000.0, "f32"),                # the smallest head width, one tile
    (1, 21, 2, 256, 5, 10000.0, "f32"),             # the widest head
    (2, 50, 4, 64, 1_000_000, 10000.0, "f32"),      # angles of 1e6 radians
    (1, 20, 2, 128, 2_000_000_000, 10000.0, "f32"),  # positions past 2^31 - 1 within the call
    (2, 33, 2, 128, 17, 500000.0, "f32"),           # another base
    (3, 70, 4, 128, 0, 10000.0, "bf16"),
    (1, 9, 16, 64, 4096, 10000.0, "bf16"),
    (2, 23, 5, 24, 3, 10000.0, "f32"),              # R / 4 = 6 vectors per row: 4 spare threads per CTA
    (1, 31, 7, 40, 11, 10000.0, "bf16"),            # R / 8 = 5 vectors per row: 1 spare thread per CTA
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}N{}H{}R{}p{}b{:g}{}".format(*c))
def test_rope_matches_oracle(case):
    B, N, H, R, pos0, base, dt = case
    q, k = _x(B, N, H, R, 90 + N, dt), _x(B, N, H, R, 91 + N, dt)
    qd, kd = q.cuda(), k.cuda()
    binding.ida_rope(qd, kd, pos0=pos0, base=base)
    torch.cuda.synchronize()
    _check(qd, ro.rope(q.double().numpy(), pos0, base), q, dt)
    _check(kd, ro.rope(k.double().numpy(), pos0, base), k, dt)


def test_rope_without_k_rotates_q_only():
    q = _x(1, 30, 2, 32, 5, "f32")
    qd = q.cuda()
    binding.ida_rope(qd, None, pos0=3)
    torch.cuda.synchronize()
    _check(qd, ro.rope(q.double().numpy(), 3), q, "f32")


def test_rope_of_zero_rows_is_a_noop():
    q = torch.empty((2, 0, 3, 32), device="cuda")
    binding.ida_rope(q, q.clone())
    torch.cuda.synchronize()
    assert binding.ida_device_error() == 0


def test_rope_in_two_calls_equals_one():
    """Rotating positions [0, n) and then [n, N) with pos0 = n equals one call over N."""
    x = _x(2, 45, 3, 64, 6, "f32")
    one, two = x.cuda(), x.cuda()
    binding.ida_rope(one, None, pos0=0)
    a, b = two[:, :19].contiguous(), two[:, 19:].contiguous()
    binding.ida_rope(a, None, pos0=0)
    binding.ida_rope(b, None, pos0=19)
    torch.cuda.synchronize()
    assert torch.equal(one, torch.cat([a, b], 1))


def test_rope_at_the_full_prefill_size_on_sampled_positions():
    """q and k of the 1.3B-like prefill ([4, 4096, 16, 128] bf16), rotated in one call as
    the benchmark does; positions sampled across the sequence, the tile edges and the
    end are checked against the oracle row by row."""
    w = configs.PREFILL_1P3B
    q, k = _x(w.B, w.N, w.H, w.R, 31, "bf16"), _x(w.B, w.N, w.H, w.R, 32, "bf16")
    qd, kd = q.cuda(), k.cuda()
    binding.ida_rope(qd, kd)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    ts = sorted(set(rng.integers(0, w.N, 24).tolist()) | {0, 7, 8, w.N - 9, w.N - 1})
    for t in ts:
        for src, dev in ((q, qd), (k, kd)):
            ref = ro.rope(src[:, t:t + 1].double().numpy(), t)
            _check(dev[:, t:t + 1], ref, src[:, t:t + 1], "bf16")
