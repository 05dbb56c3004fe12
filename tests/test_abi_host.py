"""C ABI checks that need no GPU: symbols, state size, argument validation.

Every call here is rejected by the host-side checks before the library
touches CUDA, so it runs on a machine without a GPU.
"""
import ctypes
import re
from pathlib import Path

import numpy as np
import pytest
import torch

from linear_token_mixer_sc_gb300 import binding, build

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared_symbols():
    text = (ROOT / "include" / "ida.h").read_text()
    return sorted(set(re.findall(r"IDA_API\s+[\w\s\*]*?\b(ida_\w+)\s*\(", text)))


def test_header_declares_the_exported_api():
    assert set(_declared_symbols()) == set(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_state_floats(lib):
    for d, R, M, W in [(32, 32, 16, 4), (128, 128, 64, 4), (64, 64, 64, 1), (24, 16, 15, 3)]:
        n = 2 * M * (R + d) + 2 * M + 2 * (W - 1) * R
        assert binding.ida_state_floats(d, R, M, W) == (n + 3) // 4 * 4
    assert binding.ida_state_floats(0, 32, 16, 4) == 0


def test_status_strings(lib):
    for s in range(5):
        assert binding.ida_status_str(s).startswith("IDA_")


class _Bufs:
    """Aligned host buffers standing in for device pointers (never dereferenced)."""

    def __init__(self):
        self.mem = np.zeros(64, dtype=np.float32)
        base = self.mem.ctypes.data
        self.p = ctypes.c_void_p((base + 15) // 16 * 16)
        self.mis = ctypes.c_void_p((base + 15) // 16 * 16 + 4)


def _fwd(lib, b, B=1, H=2, N=8, d=32, R=32, M=16, dtype=0, W=4, flags=0, **over):
    args = dict(q=b.p, k=b.p, v=b.p, cw=b.p, nw=b.p, bs=b.p, lam=b.p, bv=b.p, out=b.p, fs=None)
    args.update(over)
    return lib.ida_forward(args["q"], args["k"], args["v"], args["cw"], args["nw"], args["bs"],
                           args["lam"], args["bv"], args["out"], args["fs"], B, H, N, d, R, M,
                           dtype, W, flags, None)


def _dec(lib, b, B=1, H=2, d=32, R=32, M=16, dtype=0, W=4, flags=0, **over):
    args = dict(q=b.p, k=b.p, v=b.p, cw=b.p, nw=b.p, bs=b.p, lam=b.p, bv=b.p, st=b.p, out=b.p)
    args.update(over)
    return lib.ida_decode_step(args["q"], args["k"], args["v"], args["cw"], args["nw"],
                               args["bs"], args["lam"], args["bv"], args["st"], args["out"],
                               B, H, d, R, M, dtype, W, flags, None)


def test_forward_rejects_bad_arguments(lib):
    b = _Bufs()
    assert _fwd(lib, b, q=None) == binding.IDA_ERR_ARG
    assert _fwd(lib, b, out=None) == binding.IDA_ERR_ARG
    assert _fwd(lib, b, lam=b.mis) == binding.IDA_ERR_ARG
    assert _fwd(lib, b, fs=b.mis) == binding.IDA_ERR_ARG
    assert _fwd(lib, b, N=-1) == binding.IDA_ERR_ARG
    assert _fwd(lib, b, B=-2) == binding.IDA_ERR_ARG
    assert _fwd(lib, b, dtype=7) == binding.IDA_ERR_ARG
    assert _fwd(lib, b, flags=4) == binding.IDA_ERR_ARG  # no such flag bit
    assert _fwd(lib, b, M=0) == binding.IDA_ERR_ARG
    assert "pointer" in binding.ida_last_error() or "must" in binding.ida_last_error()


def _fwd_host(lib, b, B=1, H=2, N=8, d=32, R=32, M=16, dtype=0, W=4, flags=0, **over):
    args = dict(q=b.p, k=b.p, v=b.p, cw=b.p, nw=b.p, bs=b.p, lam=b.p, bv=b.p, si=None, out=b.p, fs=None,
                stg=b.p, nstg=1 << 30)
    args.update(over)
    return lib.ida_forward_host(args["q"], args["k"], args["v"], args["cw"], args["nw"], args["bs"],
                                args["lam"], args["bv"], args["si"], args["out"], args["fs"], B, H, N, d, R,
                                M, dtype, W, flags, args["stg"], args["nstg"], None)


def test_forward_host_rejects_bad_arguments_on_the_host(lib):
    """Argument errors of the host-memory prefill are found before any CUDA call."""
    b = _Bufs()
    assert _fwd_host(lib, b, q=None) == binding.IDA_ERR_ARG
    assert _fwd_host(lib, b, out=None) == binding.IDA_ERR_ARG
    assert _fwd_host(lib, b, lam=b.mis) == binding.IDA_ERR_ARG
    assert _fwd_host(lib, b, stg=None) == binding.IDA_ERR_ARG
    assert _fwd_host(lib, b, stg=b.mis) == binding.IDA_ERR_ARG
    assert "staging" in binding.ida_last_error()
    assert _fwd_host(lib, b, si=b.p, fs=b.p) == binding.IDA_ERR_ARG  # state_in overlaps final_state
    assert _fwd_host(lib, b, N=-1) == binding.IDA_ERR_ARG
    assert _fwd_host(lib, b, dtype=3) == binding.IDA_ERR_ARG
    assert _fwd_host(lib, b, R=264) == binding.IDA_ERR_UNSUPPORTED
    assert _fwd_host(lib, b, B=0) == binding.IDA_OK
    assert _fwd_host(lib, b, N=0, q=None, out=None) == binding.IDA_OK  # nothing to do without final_state


def test_forward_host_staging_bytes_without_work_or_device(lib):
    assert lib.ida_forward_host_staging_bytes(0, 2, 64, 64, 64, 64, 1, 4, 0) == 0
    assert lib.ida_forward_host_staging_bytes(1, 2, 64, 64, 64, 64, 9, 4, 0) == 0  # bad dtype
    if not torch.cuda.is_available():
        assert lib.ida_forward_host_staging_bytes(1, 2, 4096, 64, 64, 64, 1, 4, 0) == 0


def test_forward_rejects_unsupported_shapes(lib):
    b = _Bufs()
    for over in (dict(R=264), dict(d=12), dict(R=4), dict(M=129), dict(W=5), dict(d=512)):
        assert _fwd(lib, b, **over) == binding.IDA_ERR_UNSUPPORTED, over


def test_forward_empty_work_is_a_noop(lib):
    b = _Bufs()
    assert _fwd(lib, b, N=0) == binding.IDA_OK
    assert _fwd(lib, b, B=0) == binding.IDA_OK
    assert _fwd(lib, b, H=0, q=None, out=None) == binding.IDA_OK


def test_decode_rejects_bad_arguments(lib):
    b = _Bufs()
    assert _dec(lib, b, st=None) == binding.IDA_ERR_ARG
    assert _dec(lib, b, st=b.mis) == binding.IDA_ERR_ARG
    assert _dec(lib, b, dtype=3) == binding.IDA_ERR_ARG
    assert _dec(lib, b, R=100) == binding.IDA_ERR_UNSUPPORTED
    assert _dec(lib, b, B=0) == binding.IDA_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "LIB_PATH", tmp_path / "missing.so")
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        binding.load()


def _from(lib, b, sin, fs, B=1, H=2, N=8, d=32, R=32, M=16, dtype=0, W=4, flags=0):
    return lib.ida_forward_from(b.p, b.p, b.p, b.p, b.p, b.p, b.p, b.p, sin, b.p, fs, B, H, N, d, R, M,
                                dtype, W, flags, None, 0, None)


def test_forward_from_rejects_bad_states(lib):
    """ida_forward_from: a misaligned start state, or one overlapping final_state, is refused
    before any device work."""
    S = binding.ida_state_floats(32, 32, 16, 4)
    mem = np.zeros(4 * 2 * S + 64, dtype=np.float32)
    base = (mem.ctypes.data + 15) // 16 * 16
    b = _Bufs()
    p0 = ctypes.c_void_p(base)
    assert _from(lib, b, ctypes.c_void_p(base + 4), None) == binding.IDA_ERR_ARG
    assert "state_in" in binding.ida_last_error()
    # the same buffer, and a start state ending inside the final state (2 units x S floats each)
    assert _from(lib, b, p0, p0) == binding.IDA_ERR_ARG
    assert "overlap" in binding.ida_last_error()
    assert _from(lib, b, ctypes.c_void_p(base + 16 * ((S * 4) // 16)), p0) == binding.IDA_ERR_ARG
    assert _from(lib, b, p0, p0, flags=4) == binding.IDA_ERR_ARG  # no such flag bit


def test_selftest_rejects_bad_limits(lib):
    """The bounded-wait self-test checks its limit on the host, before touching CUDA."""
    for bad in (0, -5, 5_000_000_000):
        assert lib.ida_selftest_bounded_wait(bad, None) == binding.IDA_ERR_ARG


def test_backward_workspace_bytes(lib):
    """Feature rows and their gradients, a checkpoint of the state every chunk of positions
    (16 in fp32 arithmetic for bf16 inputs, 8 in fp64 for fp32 inputs), one chunk of replayed
    states per unit, plus per-tile partials: host arithmetic only."""
    n = binding.ida_backward_workspace_bytes(2, 3, 100, 32, 32, 16, binding.IDA_BF16, 4)
    assert n > 0 and n % 16 == 0
    n32 = binding.ida_backward_workspace_bytes(2, 3, 100, 32, 32, 16, binding.IDA_F32, 4)
    assert n32 > n and n32 % 32 == 0  # fp64 elements
    assert binding.ida_backward_workspace_bytes(2, 3, 200, 32, 32, 16, binding.IDA_BF16, 4) > n
    assert binding.ida_backward_workspace_bytes(2, 3, 0, 32, 32, 16, binding.IDA_BF16, 4) == 0
    assert binding.ida_backward_workspace_bytes(2, 3, 100, 32, 32, 200, binding.IDA_BF16, 4) == 0


def test_backward_rejects_bad_arguments_on_the_host(lib):
    b = _Bufs()
    p, mis = b.p, b.mis
    args = [p] * 17
    ok = dict(B=1, H=2, N=8, d=32, R=32, M=16, dtype=1, W=4, flags=0)

    def call(ptrs, ws=None, ws_bytes=0, **over):
        kw = dict(ok, **over)
        return lib.ida_backward(*ptrs, kw["B"], kw["H"], kw["N"], kw["d"], kw["R"], kw["M"], kw["dtype"],
                                kw["W"], kw["flags"], ws, ws_bytes, None)

    for i in range(17):
        bad = list(args)
        bad[i] = None
        assert call(bad) == binding.IDA_ERR_ARG
        bad[i] = mis
        assert call(bad) == binding.IDA_ERR_ARG
    # missing or short workspace
    assert call(args) == binding.IDA_ERR_ARG
    assert call(args, ws=p, ws_bytes=16) == binding.IDA_ERR_ARG
    assert call(args, B=-1) == binding.IDA_ERR_ARG
    assert call(args, flags=binding.IDA_PATH_SEQUENTIAL) == binding.IDA_ERR_ARG
    assert call(args, M=200) == binding.IDA_ERR_UNSUPPORTED
    assert call(args, W=5) == binding.IDA_ERR_UNSUPPORTED


def test_rope_rejects_bad_arguments_on_the_host(lib):
    b = _Bufs()
    p, mis = b.p, b.mis
    F = ctypes.c_float

    def call(q=p, k=None, B=1, N=8, H=2, R=32, pos0=0, base=10000.0, dtype=binding.IDA_BF16):
        return lib.ida_rope(q, k, B, N, H, R, pos0, F(base), dtype, None)

    assert call(q=None) == binding.IDA_ERR_ARG
    assert call(q=mis) == binding.IDA_ERR_ARG
    assert call(k=mis) == binding.IDA_ERR_ARG
    assert call(k=p) == binding.IDA_ERR_ARG            # k aliasing q
    assert call(B=-1) == binding.IDA_ERR_ARG
    assert call(pos0=-1) == binding.IDA_ERR_ARG
    for base in (1.0, 0.5, -3.0, float("nan"), float("inf")):
        assert call(base=base) == binding.IDA_ERR_ARG, base
    assert call(dtype=7) == binding.IDA_ERR_ARG
    for R in (4, 12, 264):
        assert call(R=R) == binding.IDA_ERR_UNSUPPORTED, R
    assert call(H=1 << 20, R=256) == binding.IDA_ERR_UNSUPPORTED
    # no rows: nothing to do, no pointer read, no CUDA call
    assert call(q=None, N=0) == binding.IDA_OK
    assert call(q=None, B=0) == binding.IDA_OK
