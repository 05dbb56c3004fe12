"""GPU parity of ida_decode_step against the fp64 CPU oracle.

The decode kernel is checked on its own (starting from the oracle's state
rounded to fp32), chained after a GPU prefill, and at the full recurrent
decode workload (batch 256, 16 heads, R = d = 128, M = 64: a 4096-position
prefill then 512 steps) on 64 (b,h) units spread over the batch.
"""
import numpy as np
import pytest
import torch

from linear_token_mixer_sc_gb300 import binding, build, configs, inputs
from oracle import ida_oracle as orc
from tests.helpers import (BF16_REL_L2, F32_MAX_ABS, F32_REL_L2,
                           max_abs_beyond_rounding, problem,
                           rel_l2, to_np, unpadded_state)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _pad_state(st64: np.ndarray, S: int) -> torch.Tensor:
    B, H, n = st64.shape
    out = np.zeros((B, H, S), dtype=np.float32)
    out[..., :n] = st64
    return torch.from_numpy(out).cuda()


@pytest.mark.parametrize("shape", [(1, 2, 32, 32, 16, 4, "f32"), (3, 2, 24, 40, 7, 3, "f32"),
                                   (2, 3, 128, 128, 64, 4, "bf16"), (1, 1, 256, 256, 128, 4, "f32"),
                                   (2, 2, 16, 8, 5, 1, "f32")],
                         ids=lambda s: "B{}H{}d{}R{}M{}W{}{}".format(*s))
@pytest.mark.parametrize("eta", [0, binding.IDA_READOUT_ETA, binding.IDA_FEAT_L2,
                                 binding.IDA_READOUT_ETA | binding.IDA_FEAT_L2])
def test_decode_from_oracle_state(shape, eta):
    """Decode kernel alone: same fp32 state in, compare out and state over 6 steps."""
    B, H, d, R, M, W, dt = shape
    N0 = 11
    q, k, v, p = problem(B, N0, H, R, d, M, W, dt, seed=200 + d)
    ref = orc.forward(q, k, v, p, flags=eta, final_state=True)
    S = binding.ida_state_floats(d, R, M, W)
    # the device starts from the oracle's state rounded to fp32; so does the oracle
    st32 = ref["final_state"].astype(np.float32)
    st_dev = _pad_state(st32, S)
    st_ref = st32.astype(np.float64)
    pd = binding.params_to_device(p)
    for step in range(6):
        qt, kt, vt = inputs.make_tokens(B, H, R, d, dt, seed=7, step=step)
        out = binding.ida_decode_step(qt.cuda(), kt.cuda(), vt.cuda(), pd, st_dev, flags=eta)
        r = orc.decode_step(qt, kt, vt, p, st_ref, flags=eta)
        st_ref[:] = st_ref.astype(np.float32)  # the state is stored as fp32 between steps
        torch.cuda.synchronize()
        got = to_np(out)
        if dt == "f32":
            assert rel_l2(got, r["out"]) <= F32_REL_L2 and max_abs_beyond_rounding(got, r["out"]) <= F32_MAX_ABS
        else:
            assert rel_l2(got, r["out"]) <= BF16_REL_L2
    got_st = unpadded_state(to_np(st_dev), d, R, M, W)
    assert rel_l2(got_st, st_ref) <= 1e-5
    assert binding.ida_device_error() == 0


def test_prefill_then_decode_chain_tiny():
    """GPU prefill(N-j) + j GPU decode steps == oracle prefill(N-j) + j oracle
    decode steps, with the state rounded to its fp32 storage format between
    calls as the library stores it."""
    w = configs.TINY_F32
    q, k, v, p = problem(w.B, w.N, w.H, w.R, w.d, w.M, w.W, w.dtype, w.seed)
    j = 9
    N = w.N
    pd = binding.params_to_device(p)
    _, st = binding.ida_forward(q[:, :N - j].contiguous().cuda(), k[:, :N - j].contiguous().cuda(),
                                v[:, :N - j].contiguous().cuda(), pd, final_state=True)
    ref = orc.forward(q[:, :N - j], k[:, :N - j], v[:, :N - j], p, final_state=True)
    st_ref = ref["final_state"].astype(np.float32).astype(np.float64)
    full = orc.forward(q, k, v, p, final_state=True)
    for i in range(N - j, N):
        out = binding.ida_decode_step(q[:, i].contiguous().cuda(), k[:, i].contiguous().cuda(),
                                      v[:, i].contiguous().cuda(), pd, st)
        r = orc.decode_step(q[:, i], k[:, i], v[:, i], p, st_ref)
        st_ref[:] = st_ref.astype(np.float32)
        got = to_np(out)
        assert rel_l2(got, r["out"]) <= F32_REL_L2 and max_abs_beyond_rounding(got, r["out"]) <= F32_MAX_ABS
        # and against the unrounded fp64 chain, at the fp32-state tolerance
        assert rel_l2(got, full["out"][:, i]) <= F32_REL_L2
    torch.cuda.synchronize()
    got_st = unpadded_state(to_np(st), w.d, w.R, w.M, w.W)
    assert rel_l2(got_st, st_ref) <= F32_REL_L2


def _decode_workload(eta, oracle_from_gpu_state):
    """Batch 256 x 16 heads: GPU prefill of 4096 positions, then 512 GPU decode steps;
    64 units (every head of four batch rows spread over the batch) checked step by step
    against the oracle.  The oracle starts from its own fp64 prefill, or from the GPU's
    state; from the GPU's state it runs twice, once rounding its state to the fp32
    storage format after every step as the library does, once keeping fp64.  Returns
    the GPU's rel-L2 over all of those outputs against the (first) oracle run, the
    worst unit, the smallest |eta denominator| / its rms seen, and the rel-L2 between
    the two oracle runs (0 without the second run)."""
    w = configs.DECODE
    dev = torch.device("cuda")
    p = inputs.make_params(w.H, w.R, w.d, w.M, w.W, w.seed)
    pd = binding.params_to_device(p)
    q, k, v = inputs.make_qkv(w.B, w.N, w.H, w.R, w.d, w.dtype, w.seed, device=dev)
    _, st = binding.ida_forward(q, k, v, pd, final_state=True)
    rows = [0, 77, 170, 255]
    r = orc.forward(q[rows].cpu(), k[rows].cpu(), v[rows].cpu(), p, final_state=True)
    del q, k, v
    torch.cuda.synchronize()
    got = unpadded_state(to_np(st[rows]), w.d, w.R, w.M, w.W)
    assert rel_l2(got, r["final_state"]) <= BF16_REL_L2
    # separate copies (the oracle updates its state argument in place)
    ref_state = np.array(got, dtype=np.float64, order="C", copy=True) if oracle_from_gpu_state else r["final_state"]
    st64 = np.array(got, dtype=np.float64, order="C", copy=True) if oracle_from_gpu_state else None
    outs, refs, refs64, dens = [], [], [], []
    for step in range(w.decode_steps):
        qt, kt, vt = inputs.make_tokens(w.B, w.H, w.R, w.d, w.dtype, w.seed, step, device=dev)
        out = binding.ida_decode_step(qt, kt, vt, pd, st, flags=eta)
        outs.append(to_np(out)[rows])
        qc, kc, vc = qt[rows].cpu(), kt[rows].cpu(), vt[rows].cpu()
        ro = orc.decode_step(qc, kc, vc, p, ref_state, flags=eta)
        if oracle_from_gpu_state:
            ref_state[:] = ref_state.astype(np.float32)
            refs64.append(orc.decode_step(qc, kc, vc, p, st64, flags=eta)["out"])
        dens.append(ro["den"])
        refs.append(ro["out"])
    assert binding.ida_device_error() == 0
    o, ref = np.stack(outs), np.stack(refs)
    per_unit = np.sqrt(((o - ref) ** 2).sum((0, 3)) / (ref ** 2).sum((0, 3)))
    worst = np.unravel_index(np.argmax(per_unit), per_unit.shape)
    den = np.stack(dens)
    den_ratio = float((np.abs(den) / np.sqrt((den ** 2).mean(axis=0))).min()) if eta else None
    fmt = rel_l2(ref, np.stack(refs64)) if oracle_from_gpu_state else 0.0
    return rel_l2(o, ref), ((rows[worst[0]], int(worst[1])), float(per_unit.max())), den_ratio, fmt, ref


def test_decode_full_workload():
    """The denominator-free readout end to end: GPU prefill then GPU decode against the
    oracle's own fp64 prefill and decode."""
    total, worst, _, _, _ = _decode_workload(0, oracle_from_gpu_state=False)
    assert total <= BF16_REL_L2, (total, worst)


def test_decode_full_workload_eta_from_gpu_state():
    """The eta readout at full scale, from the GPU's own state.  Its denominator
    Re(xi(q)^T U^T eta) cancels at some positions of this workload to a few millionths
    of its rms, where the rounding of the fp32 state alone moves the outputs: the bar is
    the stated 3e-3, or, where the data make the outputs that sensitive, the bf16
    output-rounding floor plus three times the spread between two oracle runs that
    differ only in rounding their state to fp32 after every step (the library's own
    fp32 update rounds differently from the oracle's rounded fp64 one)."""
    total, worst, den_ratio, fmt, ref = _decode_workload(binding.IDA_READOUT_ETA, oracle_from_gpu_state=True)
    floor = rel_l2(torch.from_numpy(ref).to(torch.bfloat16).double().numpy(), ref)
    bar = max(BF16_REL_L2, floor + 3 * fmt)
    print(f"eta decode: rel-L2 {total:.4g}, bf16 floor {floor:.4g}, fp32-state spread {fmt:.4g}, "
          f"min |den|/rms {den_ratio:.3g}, worst unit {worst}")
    assert total <= bar, (total, floor, fmt, worst, den_ratio)
