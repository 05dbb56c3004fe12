"""GPU parity of ida_forward_host (prefill from host memory, sliced along the sequence and
pipelined over three streams) against the fp64 oracle, and its agreement with the
device-memory entry points.

Slicing carries the state from slice to slice exactly as ida_forward_from resumes a
sequence, so the bar is the prefill's own: bf16 rel-L2 against the oracle.  Where a call
runs as one slice (the eta readout, fp32, sequential path), its bytes equal ida_forward's.
"""
import pytest
import torch

from linear_token_mixer_sc_gb300 import binding, build, configs, inputs
from oracle import ida_oracle as orc
from tests.helpers import BF16_REL_L2, F32_REL_L2, problem, rel_l2, to_np, unpadded_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _host(q, k, v, pd, pinned=True, **kw):
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    out, fs = binding.ida_forward_host(q, k, v, pd, **kw)
    torch.cuda.synchronize()
    assert binding.ida_device_error() == 0
    return out, fs


# (B, N, H, R, d, M, W, dtype, flags): several slices with a ragged last one, one slice
HOST_CASES = [
    (2, 64 * 17 + 11, 2, 64, 64, 64, 4, "bf16", 0),        # 3 slices: 512, 512, 75
    (1, 64 * 40 + 5, 2, 128, 128, 64, 4, "bf16", 0),       # 6 slices of 512, the last 5 long
    (3, 64 * 20, 2, 128, 64, 64, 3, "bf16", 0),            # slices of 512, 512, 256
    (1, 300, 3, 64, 64, 64, 4, "bf16", 0),                 # too short to slice
    (2, 64 * 18, 2, 64, 64, 64, 4, "bf16", binding.IDA_READOUT_ETA),  # eta: one slice
    (1, 90, 2, 32, 32, 16, 4, "f32", 0),                   # fp32: one slice
    (9, 64 * 16 + 9, 2, 64, 64, 64, 4, "bf16", 0),         # many rows: 3 slices, 512, 512, 9
    (4, 64 * 5 + 3, 3, 128, 128, 64, 2, "bf16", 0),        # many rows, one slice
    (9, 70, 2, 64, 64, 64, 4, "bf16", binding.IDA_READOUT_ETA),  # eta, many rows: one slice
    (2, 64 * 17 + 11, 2, 128, 128, 64, 4, "bf16", binding.IDA_FEAT_L2),  # l_2 map, 3 resumed slices
]


@pytest.mark.parametrize("case", HOST_CASES, ids=lambda c: "B{}N{}H{}R{}d{}M{}W{}{}f{}".format(*c))
def test_host_prefill_matches_oracle(case):
    B, N, H, R, d, M, W, dt, flags = case
    q, k, v, p = problem(B, N, H, R, d, M, W, dt, seed=500 + N)
    pd = binding.params_to_device(p)
    out, fs = _host(q, k, v, pd, final_state=True, flags=flags)
    ref = orc.forward(q, k, v, p, flags=flags & (binding.IDA_READOUT_ETA | binding.IDA_FEAT_L2), final_state=True)
    tol = F32_REL_L2 if dt == "f32" else BF16_REL_L2
    assert rel_l2(to_np(out), ref["out"]) <= tol
    assert rel_l2(unpadded_state(to_np(fs), d, R, M, W), ref["final_state"]) <= tol


@pytest.mark.parametrize("B", [2, 5])
def test_host_prefill_from_state_matches_oracle(B):
    """A host call resumed from a state (several slices) against the oracle run from that state."""
    N1, N2, H, R, d, M, W = 150, 64 * 19 + 3, 2, 64, 64, 64, 4
    q, k, v, p = problem(B, N1 + N2, H, R, d, M, W, "bf16", seed=77)
    pd = binding.params_to_device(p)
    dev = torch.device("cuda")
    _, fs1 = binding.ida_forward(q[:, :N1].contiguous().to(dev), k[:, :N1].contiguous().to(dev),
                                 v[:, :N1].contiguous().to(dev), pd, final_state=True)
    torch.cuda.synchronize()
    st_in = fs1.cpu()
    out, fs = _host(q[:, N1:].contiguous(), k[:, N1:].contiguous(), v[:, N1:].contiguous(), pd,
                    final_state=True, state_in=st_in)
    ref = orc.forward(q[:, N1:], k[:, N1:], v[:, N1:], p, final_state=True,
                      state_in=unpadded_state(to_np(fs1), d, R, M, W))
    assert rel_l2(to_np(out), ref["out"]) <= BF16_REL_L2
    assert rel_l2(unpadded_state(to_np(fs), d, R, M, W), ref["final_state"]) <= BF16_REL_L2
    full = orc.forward(q, k, v, p)
    assert rel_l2(to_np(out), full["out"][:, N1:]) <= BF16_REL_L2


@pytest.mark.parametrize("B", [2, 9])
def test_host_sequential_path_equals_device_call_bytewise(B):
    """A call the tensor-core path does not take (eta readout) runs as one slice: its bytes
    are ida_forward's."""
    q, k, v, p = problem(B, 64 * 18, 2, 64, 64, 64, 4, "bf16", seed=78)
    pd = binding.params_to_device(p)
    flags = binding.IDA_READOUT_ETA
    out_h, fs_h = _host(q, k, v, pd, final_state=True, flags=flags)
    dev = torch.device("cuda")
    out_d, fs_d = binding.ida_forward(q.to(dev), k.to(dev), v.to(dev), pd, flags=flags, final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu())
    assert torch.equal(fs_h, fs_d.cpu())


@pytest.mark.parametrize("B", [2, 5])
def test_host_pageable_memory_gives_the_same_bytes(B):
    q, k, v, p = problem(B, 64 * 17 + 11, 2, 64, 64, 64, 4, "bf16", seed=79)
    pd = binding.params_to_device(p)
    a, fa = _host(q, k, v, pd, pinned=True, final_state=True)
    b, fb = _host(q, k, v, pd, pinned=False, out=torch.empty_like(a), final_state=torch.empty_like(fa))
    assert torch.equal(a, b)
    assert torch.equal(fa, fb)


def test_host_repeated_calls_are_deterministic():
    q, k, v, p = problem(1, 64 * 40 + 5, 2, 128, 128, 64, 4, "bf16", seed=80)
    pd = binding.params_to_device(p)
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    staging = torch.empty(binding.ida_forward_host_staging_bytes(1, 2, 64 * 40 + 5, 128, 128, 64,
                                                                 binding.IDA_BF16, 4), dtype=torch.uint8,
                          device="cuda")
    outs = []
    for _ in range(3):
        out, _ = binding.ida_forward_host(q, k, v, pd, staging=staging)
        torch.cuda.synchronize()
        outs.append(out)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_host_call_is_ordered_on_a_side_stream():
    """Issued on a non-default stream, the call runs after the work queued there before it
    (a fill of the staging buffer, which the call must overwrite) and is complete once that
    stream alone is synchronised."""
    q, k, v, p = problem(1, 64 * 20, 2, 64, 64, 64, 4, "bf16", seed=81)
    pd = binding.params_to_device(p)
    ref, _ = _host(q, k, v, pd)
    s = torch.cuda.Stream()
    staging = torch.empty(binding.ida_forward_host_staging_bytes(1, 2, 64 * 20, 64, 64, 64,
                                                                 binding.IDA_BF16, 4), dtype=torch.uint8,
                          device="cuda")
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    with torch.cuda.stream(s):
        staging.fill_(0xFF)  # queued before the call: NaN patterns the call must overwrite
        out, _ = binding.ida_forward_host(q, k, v, pd, staging=staging, stream=s)
    s.synchronize()
    assert torch.equal(out, ref)


@pytest.mark.parametrize("B", [1, 6])
def test_host_zero_length_copies_state(B):
    q, k, v, p = problem(B, 9, 2, 64, 64, 64, 4, "bf16", seed=82)
    pd = binding.params_to_device(p)
    _, fs1 = _host(q, k, v, pd, final_state=True)
    e = torch.empty((B, 0, 2, 64), dtype=torch.bfloat16)
    _, fs2 = _host(e, e.clone(), e.clone(), pd, final_state=True, state_in=fs1)
    assert torch.equal(fs1, fs2)
    _, fs3 = _host(e, e.clone(), e.clone(), pd, final_state=torch.full_like(fs1, 3.0))
    assert torch.count_nonzero(fs3).item() == 0


def test_host_rejects_small_staging():
    q, k, v, p = problem(1, 64 * 20, 2, 64, 64, 64, 4, "bf16", seed=83)
    pd = binding.params_to_device(p)
    with pytest.raises(binding.IdaError, match="staging"):
        binding.ida_forward_host(q, k, v, pd, staging=torch.empty(1024, dtype=torch.uint8, device="cuda"))


def test_host_prefill_at_the_full_1p3b_size():
    """The 1.3B-like prefill ([4, 4096, 16, 128] bf16, 8 slices of 512) from pinned host
    memory, as the benchmark's end-to-end leg runs it: against the device call on the whole
    output, and against the oracle on sampled units."""
    w = configs.PREFILL_1P3B
    p = inputs.make_params(w.H, w.R, w.d, w.M, w.W, w.seed)
    q, k, v = inputs.make_qkv(w.B, w.N, w.H, w.R, w.d, w.dtype, w.seed)
    pd = binding.params_to_device(p)
    out_h, _ = _host(q, k, v, pd)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out_d, _ = binding.ida_forward(qd, kd, vd, pd, workspace=binding.forward_workspace(qd, vd, pd, 0))
    torch.cuda.synchronize()
    assert rel_l2(to_np(out_h), to_np(out_d)) <= BF16_REL_L2
    units = [0, 17, 38, 63]
    ref = orc.forward(q, k, v, p, units=units)
    for u in units:
        b, h = divmod(u, w.H)
        assert rel_l2(to_np(out_h)[b, :, h], ref["out"][b, :, h]) <= BF16_REL_L2, u
