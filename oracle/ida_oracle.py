"""ctypes wrapper around the fp64 CPU oracle (``ida_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the CPU-baseline
leg of ``bench.py`` are the only callers.  The CUDA library never loads this
module and this module never loads the CUDA library; the two sides meet only
at the seeded input generator.

Every function here marshals arguments and calls the C code; no arithmetic of
the mixer lives in Python.  See ``ida_oracle.c`` for what each step computes
and which passage of "Interdomain Attention: Beyond Token-Level Key-Value
Memory" it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from pathlib import Path

import numpy as np
import torch

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "ida_oracle.c"
_LIB_PATH = _HERE / "liboracle_ida.so"
_lock = threading.Lock()
_lib = None

READOUT_ETA = 1
FEAT_L2 = 2  # the "SiLU/l_2" reading of the feature map
F32, BF16 = 0, 1

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_ip = ctypes.POINTER(ctypes.c_int)
_vp = ctypes.c_void_p
_i = ctypes.c_int


def build(force: bool = False) -> Path:
    """Compile the oracle with gcc (portable C11 + OpenMP, no arch flags)."""
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC",
             str(_SRC), "-o", str(tmp), "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(str(_LIB_PATH))
            L.orc_state_doubles.restype = ctypes.c_size_t
            L.orc_state_doubles.argtypes = [_i, _i, _i, _i]
            L.orc_silu.restype = ctypes.c_double
            L.orc_silu.argtypes = [ctypes.c_double]
            L.orc_causal_conv.argtypes = [_dp, _i, _i, _dp, _i, _dp, _dp]
            L.orc_feature_map.argtypes = [_dp, _i, _i, _dp]
            L.orc_feature_map_l2.argtypes = [_dp, _i, _i, _dp]
            L.orc_rmsnorm_affine.argtypes = [_dp, _i, _i, _dp, _dp, _dp]
            L.orc_unit_features.argtypes = [_dp, _dp, _dp, _i, _i, _i, _i, _dp, _dp,
                                            _dp, _dp, _dp, _dp, _dp, _dp, _dp]
            L.orc_unit_forward.argtypes = [_dp, _dp, _dp, _i, _i, _i, _i, _i, _dp, _dp,
                                           _dp, _dp, _dp, _dp, _i, _dp, _dp, _dp, _dp, _dp]
            L.orc_unit_forward_chunked.argtypes = [_dp, _dp, _dp, _i, _i, _i, _i, _dp, _dp,
                                                   _i, _i, _dp, _dp, _dp]
            L.orc_forward.restype = _i
            L.orc_forward.argtypes = [_vp, _vp, _vp, _i, _fp, _fp, _fp, _fp, _fp, _dp, _dp,
                                      _dp, _i, _i, _i, _i, _i, _i, _i, _i, _ip, _i, _i]
            L.orc_forward_from.restype = _i
            L.orc_forward_from.argtypes = [_vp, _vp, _vp, _i, _fp, _fp, _fp, _fp, _fp, _dp, _dp,
                                           _dp, _dp, _i, _i, _i, _i, _i, _i, _i, _i, _ip, _i, _i]
            L.orc_decode_step.restype = _i
            L.orc_decode_step.argtypes = [_vp, _vp, _vp, _i, _fp, _fp, _fp, _fp, _fp, _dp,
                                          _dp, _dp, _i, _i, _i, _i, _i, _i, _i, _ip, _i, _i]
            L.orc_max_threads.restype = _i
            _lib = L
    return _lib


# ---- marshalling helpers -------------------------------------------------

def _d(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray | None, t=_dp):
    return None if a is None else a.ctypes.data_as(t)


def _raw(x: torch.Tensor):
    """(pointer, dtype code, keep-alive) for a CPU fp32/bf16 tensor."""
    x = x.detach().to("cpu").contiguous()
    if x.dtype == torch.bfloat16:
        return ctypes.c_void_p(x.data_ptr()), BF16, x
    if x.dtype == torch.float32:
        return ctypes.c_void_p(x.data_ptr()), F32, x
    raise TypeError(f"oracle takes fp32 or bf16 inputs, got {x.dtype}")


def _f32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def state_doubles(d: int, R: int, M: int, W: int) -> int:
    return int(lib().orc_state_doubles(d, R, M, W))


# ---- single-step building blocks (float64 in, float64 out) ---------------

def silu(x: float) -> float:
    return float(lib().orc_silu(float(x)))


def causal_conv(x, w, tail=None) -> np.ndarray:
    x, w = _d(x), _d(w)
    N, C = x.shape
    W = w.shape[1]
    s = np.empty_like(x)
    tail = None if tail is None else _d(tail)
    lib().orc_causal_conv(_ptr(x), N, C, _ptr(w), W, _ptr(tail), _ptr(s))
    return s


def feature_map(s, l2: bool = False) -> np.ndarray:
    s = _d(s)
    xi = np.empty_like(s)
    fn = lib().orc_feature_map_l2 if l2 else lib().orc_feature_map
    fn(_ptr(s), s.shape[0], s.shape[1], _ptr(xi))
    return xi


def rmsnorm_affine(x, w, b) -> np.ndarray:
    x, w, b = _d(x), _d(w), _d(b)
    y = np.empty_like(x)
    lib().orc_rmsnorm_affine(_ptr(x), x.shape[0], x.shape[1], _ptr(w), _ptr(b), _ptr(y))
    return y


def unit_features(q, k, v, wq, wk, norm_w, bias, tail_q=None, tail_k=None):
    """xi(q), kt, vt for one (b,h) unit (rows [N][R], [N][R], [N][d])."""
    q, k, v = _d(q), _d(k), _d(v)
    N, R = q.shape
    d = v.shape[1]
    W = np.asarray(wq).shape[1]
    xq, kt, vt = np.empty((N, R)), np.empty((N, R)), np.empty((N, d))
    tq = None if tail_q is None else _d(tail_q)
    tk = None if tail_k is None else _d(tail_k)
    lib().orc_unit_features(_ptr(q), _ptr(k), _ptr(v), N, R, d, W, _ptr(_d(wq)), _ptr(_d(wk)),
                            _ptr(_d(norm_w)), _ptr(_d(bias)), _ptr(tq), _ptr(tk),
                            _ptr(xq), _ptr(kt), _ptr(vt))
    return xq, kt, vt


def _ri(z) -> np.ndarray:
    z = np.asarray(z)
    if np.iscomplexobj(z):
        return _d(np.stack([z.real, z.imag], axis=-1))
    return _d(z)


def unit_forward(q, k, v, wq, wk, norm_w, bias, lam, Bv, flags=0, state=None,
                 tail_q=None, tail_k=None):
    """Step recurrence for one unit.  lam/Bv: complex [M] or [M,2] (re,im).

    Returns (out [N][d], den [N], state [2M(R+d)+2M]).  ``state`` (if given)
    is the starting planar state + eta; it is not modified.
    """
    q, k, v = _d(q), _d(k), _d(v)
    N, R = q.shape
    d = v.shape[1]
    W = np.asarray(wq).shape[1]
    lam, Bv = _ri(lam), _ri(Bv)
    M = lam.shape[0]
    st = np.zeros(2 * M * (R + d) + 2 * M) if state is None else _d(state).copy()
    out, den = np.empty((N, d)), np.empty(N)
    tq = None if tail_q is None else _d(tail_q)
    tk = None if tail_k is None else _d(tail_k)
    lib().orc_unit_forward(_ptr(q), _ptr(k), _ptr(v), N, R, d, M, W, _ptr(_d(wq)), _ptr(_d(wk)),
                           _ptr(_d(norm_w)), _ptr(_d(bias)), _ptr(lam), _ptr(Bv), int(flags),
                           _ptr(st), _ptr(tq), _ptr(tk), _ptr(out), _ptr(den))
    return out, den, st


def unit_forward_chunked(xq, kt, vt, lam, Bv, C, flags=0, state=None):
    """Chunked re-association of the recurrence on prepared features."""
    xq, kt, vt = _d(xq), _d(kt), _d(vt)
    N, R = xq.shape
    d = vt.shape[1]
    lam, Bv = _ri(lam), _ri(Bv)
    M = lam.shape[0]
    st = np.zeros(2 * M * (R + d) + 2 * M) if state is None else _d(state).copy()
    out, den = np.empty((N, d)), np.empty(N)
    lib().orc_unit_forward_chunked(_ptr(xq), _ptr(kt), _ptr(vt), N, R, d, M, _ptr(lam), _ptr(Bv),
                                   int(flags), int(C), _ptr(st), _ptr(out), _ptr(den))
    return out, den, st


# ---- batched entry points on the library's own argument layout -----------

def forward(q, k, v, params: dict, flags: int = 0, final_state: bool = False,
            units=None, nthreads: int = 0, want_den: bool = False, state_in=None):
    """Prefill of [B,N,H,*] fp32/bf16 tensors (CPU) with fp32 parameters.

    params: conv_w [2,H,R,W], norm_w [H,R+d], bias [H,R+d], lambda [H,M,2],
    Bvec [H,M,2].  state_in: optional [B,H,S] state before position 0 (planar
    X, eta, raw conv tails; S = state_doubles), zero when None.  Returns
    dict(out [B,N,H,d] float64, den [B,N,H] or None, final_state [B,H,S]
    float64 or None).  With ``units`` (ids b*H+h) only those units are
    computed; other entries stay NaN.
    """
    qp, dt, qk = _raw(q)
    kp, dt2, kk = _raw(k)
    vp, dt3, vk = _raw(v)
    assert dt == dt2 == dt3
    B, N, H, R = qk.shape
    d = vk.shape[3]
    conv_w, norm_w, bias = _f32(params["conv_w"]), _f32(params["norm_w"]), _f32(params["bias"])
    lam, Bv = _f32(params["lambda"]), _f32(params["Bvec"])
    M, W = lam.shape[1], conv_w.shape[3]
    out = np.full((B, N, H, d), np.nan)
    den = np.full((B, N, H), np.nan) if want_den or (flags & READOUT_ETA) else None
    S = state_doubles(d, R, M, W)
    fs = np.full((B, H, S), np.nan) if final_state else None
    uarr = None if units is None else np.ascontiguousarray(units, dtype=np.int32)
    sin = None
    if state_in is not None:
        sin = _d(state_in)
        assert sin.shape == (B, H, S), (sin.shape, (B, H, S))
    rc = lib().orc_forward_from(qp, kp, vp, dt, _ptr(conv_w, _fp), _ptr(norm_w, _fp),
                                _ptr(bias, _fp), _ptr(lam, _fp), _ptr(Bv, _fp), _ptr(sin),
                                _ptr(out), _ptr(fs), _ptr(den), B, H, N, d, R, M, W, int(flags),
                                _ptr(uarr, _ip), 0 if uarr is None else len(uarr), int(nthreads))
    assert rc == 0
    return {"out": out, "den": den, "final_state": fs}


def decode_step(q, k, v, params: dict, state: np.ndarray, flags: int = 0, units=None,
                nthreads: int = 0):
    """One decode step on [B,H,*] tensors; ``state`` [B,H,S] float64 updated in place."""
    qp, dt, qk = _raw(q)
    kp, _, kk = _raw(k)
    vp, _, vk = _raw(v)
    B, H, R = qk.shape
    d = vk.shape[2]
    conv_w, norm_w, bias = _f32(params["conv_w"]), _f32(params["norm_w"]), _f32(params["bias"])
    lam, Bv = _f32(params["lambda"]), _f32(params["Bvec"])
    M, W = lam.shape[1], conv_w.shape[3]
    assert state.dtype == np.float64 and state.flags.c_contiguous
    assert state.shape == (B, H, state_doubles(d, R, M, W))
    out = np.full((B, H, d), np.nan)
    den = np.full((B, H), np.nan)
    uarr = None if units is None else np.ascontiguousarray(units, dtype=np.int32)
    rc = lib().orc_decode_step(qp, kp, vp, dt, _ptr(conv_w, _fp), _ptr(norm_w, _fp),
                               _ptr(bias, _fp), _ptr(lam, _fp), _ptr(Bv, _fp), _ptr(state),
                               _ptr(out), _ptr(den), B, H, d, R, M, W, int(flags),
                               _ptr(uarr, _ip), 0 if uarr is None else len(uarr), int(nthreads))
    assert rc == 0
    return {"out": out, "den": den}


def max_threads() -> int:
    return int(lib().orc_max_threads())
