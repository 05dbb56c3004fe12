"""Robustness checks that stand in for a memory sanitizer, and the failure path.

- Guard bands: ``out`` and the state buffers are views into larger buffers
  whose margins hold a canary pattern; after each call the margins must be
  untouched (no kernel writes outside its output), and the outputs and states
  must be free of NaN and Inf.  Odd shapes (ragged lengths, d != R, odd M,
  W < 4, the largest R, d, M) on every prefill path, both readouts, and decode.
- Failure reporting: the library's bounded-wait self-test makes a wait run out
  on purpose (an mbarrier nothing arrives on, given a limit of 1e5 cycles); the
  kernel returns, records the wait-timeout code, the next call reports
  IDA_ERR_DEVICE, and the GPU keeps working.
"""
import numpy as np
import pytest
import torch

from linear_token_mixer_sc_gb300 import binding, build
from oracle import ida_oracle as orc
from tests.helpers import BF16_REL_L2, F32_REL_L2, problem, rel_l2, to_np, unpadded_state

pytestmark = pytest.mark.gpu

GUARD = 1024  # canary elements before and after each guarded buffer (16-byte multiples)
CANARY_F32 = 0x7FA5A5A5  # a NaN payload no kernel produces
CANARY_BF16 = 0x7FA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _guarded(shape, dtype):
    """A tensor of `shape` inside a buffer with canary margins: (view, whole buffer)."""
    n = int(np.prod(shape))
    if dtype == torch.float32:
        raw = torch.full((n + 2 * GUARD,), CANARY_F32, dtype=torch.int32, device="cuda")
    else:
        raw = torch.full((n + 2 * GUARD,), CANARY_BF16, dtype=torch.int16, device="cuda")
    whole = raw.view(dtype)
    return whole[GUARD:GUARD + n].view(shape), raw


def _margins_intact(raw, n):
    canary = CANARY_F32 if raw.dtype == torch.int32 else CANARY_BF16
    head, tail = raw[:GUARD], raw[GUARD + n:]
    return bool((head == canary).all()) and bool((tail == canary).all())


def _finite(t):
    return bool(torch.isfinite(t.float()).all())


PATHS = {"default": 0, "sequential": binding.IDA_PATH_SEQUENTIAL}
# (B, N, H, R, d, M, W, dtype)
SHAPES = [
    (2, 37, 3, 32, 64, 15, 4, "f32"),
    (1, 70, 2, 64, 32, 7, 2, "f32"),
    (1, 33, 1, 256, 256, 128, 4, "f32"),
    (1, 65, 3, 64, 64, 33, 4, "bf16"),
    (3, 70, 2, 128, 64, 64, 3, "bf16"),
    (1, 200, 2, 64, 128, 64, 2, "bf16"),
    (1, 64 * 9 + 5, 2, 128, 128, 64, 4, "bf16"),  # split across SMs with a workspace
]


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}N{}H{}R{}d{}M{}W{}{}".format(*s))
def test_prefill_writes_nothing_outside_its_outputs(shape, path):
    B, N, H, R, d, M, W, dt = shape
    q, k, v, p = problem(B, N, H, R, d, M, W, dt, seed=500 + N)
    dev = torch.device("cuda")
    pd = binding.params_to_device(p)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    S = binding.ida_state_floats(d, R, M, W)
    tol = F32_REL_L2 if dt == "f32" else BF16_REL_L2
    for eta in (0, binding.IDA_READOUT_ETA):
        flags = PATHS[path] | eta
        out, out_raw = _guarded((B, N, H, d), qd.dtype)
        fs, fs_raw = _guarded((B, H, S), torch.float32)
        ws = binding.forward_workspace(qd, vd, pd, flags)
        ws_raw = None
        if ws is not None:  # the workspace is guarded too
            wsv, ws_raw = _guarded((ws.numel() // 4,), torch.float32)
            ws = wsv
        binding.ida_forward(qd, kd, vd, pd, out=out, final_state=fs, flags=flags, workspace=ws)
        torch.cuda.synchronize()
        assert binding.ida_device_error() == 0
        assert _margins_intact(out_raw, out.numel()), "write outside out"
        assert _margins_intact(fs_raw, fs.numel()), "write outside final_state"
        if ws_raw is not None:
            assert _margins_intact(ws_raw, ws.numel()), "write outside the workspace"
        assert _finite(out) and _finite(fs)
        ref = orc.forward(q, k, v, p, flags=eta, final_state=True)
        assert rel_l2(to_np(out), ref["out"]) <= tol
        assert rel_l2(unpadded_state(to_np(fs), d, R, M, W), ref["final_state"]) <= tol


@pytest.mark.parametrize("shape", [(3, 2, 24, 40, 7, 3, "f32"), (2, 3, 128, 128, 64, 4, "bf16"),
                                   (1, 1, 256, 256, 128, 4, "f32"), (2, 2, 16, 8, 5, 1, "f32")],
                         ids=lambda s: "B{}H{}d{}R{}M{}W{}{}".format(*s))
def test_decode_writes_nothing_outside_its_state_and_output(shape):
    B, H, d, R, M, W, dt = shape
    q, k, v, p = problem(B, 13, H, R, d, M, W, dt, seed=600 + d)
    dev = torch.device("cuda")
    pd = binding.params_to_device(p)
    S = binding.ida_state_floats(d, R, M, W)
    st, st_raw = _guarded((B, H, S), torch.float32)
    binding.ida_forward(q.to(dev), k.to(dev), v.to(dev), pd, final_state=st)
    ref = orc.forward(q, k, v, p, final_state=True)
    st_ref = ref["final_state"].astype(np.float32).astype(np.float64)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    for step in range(3):
        qt = torch.randn(B, H, R, generator=torch.Generator().manual_seed(step)).to(tdt)
        kt = torch.randn(B, H, R, generator=torch.Generator().manual_seed(100 + step)).to(tdt)
        vt = torch.randn(B, H, d, generator=torch.Generator().manual_seed(200 + step)).to(tdt)
        out, out_raw = _guarded((B, H, d), tdt)
        binding.ida_decode_step(qt.to(dev), kt.to(dev), vt.to(dev), pd, st, out=out)
        r = orc.decode_step(qt, kt, vt, p, st_ref)
        st_ref[:] = st_ref.astype(np.float32)  # the library stores the state as fp32
        torch.cuda.synchronize()
        assert binding.ida_device_error() == 0
        assert _margins_intact(out_raw, out.numel()), "write outside out"
        assert _margins_intact(st_raw, st.numel()), "write outside state_inout"
        assert _finite(out) and _finite(st)
        assert rel_l2(to_np(out), r["out"]) <= (F32_REL_L2 if dt == "f32" else BF16_REL_L2)


def test_bounded_wait_runs_out_and_is_reported():
    """A wait given 1e5 cycles on an mbarrier nothing completes gives up, the kernel
    records the wait-timeout code (1), and the next call reports IDA_ERR_DEVICE; the
    word is then clear and the library computes correctly again."""
    assert binding.ida_device_error() == 0
    binding.ida_selftest_bounded_wait(100_000)
    torch.cuda.synchronize()
    assert binding.ida_device_error() == 1  # read and cleared
    assert binding.ida_device_error() == 0
    # the next call after a timeout reports it, once
    binding.ida_selftest_bounded_wait(100_000)
    torch.cuda.synchronize()
    q, k, v, p = problem(1, 40, 2, 64, 64, 64, 4, "bf16", seed=7)
    dev = torch.device("cuda")
    pd = binding.params_to_device(p)
    with pytest.raises(binding.IdaError) as ei:
        binding.ida_forward(q.to(dev), k.to(dev), v.to(dev), pd)
    assert ei.value.status == binding.IDA_ERR_DEVICE
    assert "device error code 1" in str(ei.value)
    assert binding.ida_device_error() == 0
    out, _ = binding.ida_forward(q.to(dev), k.to(dev), v.to(dev), pd)
    torch.cuda.synchronize()
    assert binding.ida_device_error() == 0
    assert rel_l2(to_np(out), orc.forward(q, k, v, p)["out"]) <= BF16_REL_L2
