"""ida_forward_noalloc: prefill for callers that cannot allocate device memory.

Some callers of this library may not allocate: a plug-in that its host
framework hands only input and output buffers, or a serving loop that must
not touch the allocator once running.  ida_forward_noalloc serves them with
the library's static scratch instead of a caller workspace.  This file checks,
through the C ABI, that it returns what ida_forward_ws returns with a
caller-allocated workspace, on two calls in a row (the static scratch keeps
the first call's contents when the second starts).  It is collected last so
that a run stopping at the first failure has run everything else first.
"""
import pytest
import torch

from linear_token_mixer_sc_gb300 import binding, build
from tests.helpers import BF16_REL_L2, problem, rel_l2, to_np, unpadded_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _inputs(seed, B=1, N=64 * 40 + 17, H=2, R=128, d=128):
    q, k, v, p = problem(B, N, H, R, d, 64, 4, "bf16", seed=seed)
    dev = torch.device("cuda")
    return q.to(dev), k.to(dev), v.to(dev), binding.params_to_device(p)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    calls = [_inputs(41), _inputs(42)]
    q, k, v, pd = calls[0]
    B, N, H, R = q.shape
    d = v.shape[3]
    # the shape is split into segments, so the static scratch is really used
    assert binding.ida_forward_workspace_bytes(B, H, N, d, R, 64, binding.IDA_BF16, 4) > 0
    for q, k, v, pd in calls:
        ws = binding.forward_workspace(q, v, pd)
        ref, ref_st = binding.ida_forward(q, k, v, pd, final_state=True, workspace=ws)
        out = torch.empty_like(ref)
        st = torch.empty_like(ref_st)
        binding.ida_forward_noalloc(q, k, v, pd, out, final_state=st)
        torch.cuda.synchronize()
        assert binding.ida_device_error() == 0
        assert rel_l2(to_np(out), to_np(ref)) <= BF16_REL_L2
        assert rel_l2(unpadded_state(to_np(st), d, R, 64, 4),
                      unpadded_state(to_np(ref_st), d, R, 64, 4)) <= BF16_REL_L2
