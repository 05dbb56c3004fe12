"""Python binding of the C ABI in ``include/ida.h`` (``_lib/libida.so``).

Argument marshalling only: every step of the mixer runs in the library's CUDA
kernels.  Torch supplies device memory and the stream.  There is no fallback:
if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

import torch

LIB_PATH = Path(__file__).resolve().parent / "_lib" / "libida.so"

IDA_OK, IDA_ERR_ARG, IDA_ERR_UNSUPPORTED, IDA_ERR_CUDA, IDA_ERR_DEVICE = range(5)
IDA_F32, IDA_BF16 = 0, 1
IDA_READOUT_ETA = 1
IDA_FEAT_L2 = 2
IDA_PATH_SEQUENTIAL = 256

EXPORTED = ("ida_state_floats", "ida_forward", "ida_forward_ws", "ida_forward_from", "ida_forward_workspace_bytes",
            "ida_forward_noalloc", "ida_decode_step", "ida_device_error", "ida_status_str",
            "ida_last_error", "ida_selftest_bounded_wait", "ida_backward", "ida_backward_workspace_bytes",
            "ida_forward_ideal", "ida_rope", "ida_forward_host", "ida_forward_host_staging_bytes")

_lock = threading.Lock()
_lib = None
_vp, _fp, _i = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int


class IdaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def load() -> ctypes.CDLL:
    """Load ``libida.so``; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not LIB_PATH.exists():
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with linear_token_mixer_sc_gb300.build.build()")
            L = ctypes.CDLL(str(LIB_PATH))
            L.ida_state_floats.restype = ctypes.c_size_t
            L.ida_state_floats.argtypes = [_i, _i, _i, _i]
            L.ida_forward.restype = _i
            L.ida_forward.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp, _vp, _fp,
                                      _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp]
            L.ida_forward_ws.restype = _i
            L.ida_forward_ws.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp, _vp, _fp,
                                         _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp, ctypes.c_size_t, _vp]
            L.ida_forward_from.restype = _i
            L.ida_forward_from.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp, _fp, _vp, _fp,
                                           _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp, ctypes.c_size_t, _vp]
            L.ida_forward_workspace_bytes.restype = ctypes.c_size_t
            L.ida_forward_workspace_bytes.argtypes = [_i] * 9
            L.ida_forward_host.restype = _i
            L.ida_forward_host.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp, _fp, _vp, _fp,
                                           _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp, ctypes.c_size_t, _vp]
            L.ida_forward_host_staging_bytes.restype = ctypes.c_size_t
            L.ida_forward_host_staging_bytes.argtypes = [_i] * 9
            L.ida_forward_noalloc.restype = _i
            L.ida_forward_noalloc.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp, _vp, _fp,
                                              _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp]
            L.ida_decode_step.restype = _i
            L.ida_decode_step.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp, _fp, _vp,
                                          _i, _i, _i, _i, _i, _i, _i, _i, _vp]
            L.ida_backward.restype = _i
            L.ida_backward.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp, _vp, _vp, _vp, _vp,
                                       _fp, _fp, _fp, _fp, _fp,
                                       _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp, ctypes.c_size_t, _vp]
            L.ida_backward_workspace_bytes.restype = ctypes.c_size_t
            L.ida_backward_workspace_bytes.argtypes = [_i] * 9
            L.ida_forward_ideal.restype = _i
            L.ida_forward_ideal.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _vp]
            L.ida_rope.restype = _i
            L.ida_rope.argtypes = [_vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i, _vp]
            L.ida_selftest_bounded_wait.restype = _i
            L.ida_selftest_bounded_wait.argtypes = [ctypes.c_longlong, _vp]
            L.ida_device_error.restype = _i
            L.ida_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
            L.ida_status_str.restype = ctypes.c_char_p
            L.ida_status_str.argtypes = [_i]
            L.ida_last_error.restype = ctypes.c_char_p
            L.ida_last_error.argtypes = []
            _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != IDA_OK:
        L = load()
        raise IdaError(status, f"{what}: {L.ida_status_str(status).decode()} "
                               f"({L.ida_last_error().decode()})")


def ida_state_floats(d: int, R: int, M: int, W: int) -> int:
    return int(load().ida_state_floats(d, R, M, W))


def ida_status_str(status: int) -> str:
    return load().ida_status_str(status).decode()


def ida_last_error() -> str:
    return load().ida_last_error().decode()


def ida_device_error() -> int:
    code = ctypes.c_uint(0)
    load().ida_device_error(ctypes.byref(code))
    return int(code.value)


def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return IDA_F32
    if t.dtype == torch.bfloat16:
        return IDA_BF16
    raise TypeError(f"q/k/v must be float32 or bfloat16, got {t.dtype}")


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _params(p: dict):
    out = []
    for key in ("conv_w", "norm_w", "bias", "lambda", "Bvec"):
        t = p[key]
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
            raise ValueError(f"parameter {key} must be a contiguous float32 CUDA tensor")
        out.append(t)
    return out


def ida_forward_workspace_bytes(B: int, H: int, N: int, d: int, R: int, M: int, dtype: int,
                                W: int, flags: int = 0) -> int:
    return int(load().ida_forward_workspace_bytes(B, H, N, d, R, M, dtype, W, flags))


def ida_forward_host_staging_bytes(B: int, H: int, N: int, d: int, R: int, M: int, dtype: int,
                                   W: int, flags: int = 0) -> int:
    return int(load().ida_forward_host_staging_bytes(B, H, N, d, R, M, dtype, W, flags))


def ida_forward_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, params: dict,
                     out: torch.Tensor | None = None, final_state: torch.Tensor | bool | None = None,
                     state_in: torch.Tensor | None = None, flags: int = 0,
                     staging: torch.Tensor | None = None, stream=None):
    """Prefill from host memory (``ida_forward_host``).  q, k [B,N,H,R], v [B,N,H,d]
    contiguous CPU tensors (fp32/bf16; pinned memory lets the copies overlap the
    kernels).  ``params`` as for ``ida_forward`` (CUDA).  ``out``: CPU tensor to fill,
    or None to allocate a pinned one.  ``final_state``: CPU float32 [B,H,S] tensor,
    True to allocate a pinned one, or None.  ``state_in``: CPU float32 [B,H,S] or None.
    ``staging``: CUDA tensor of at least ``ida_forward_host_staging_bytes`` bytes, or
    None to allocate one.  Asynchronous on ``stream``: synchronise it before reading
    ``out`` / ``final_state``.  Returns (out, final_state).
    """
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CPU tensors")
    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype")
    B, N, H, R = q.shape
    d = v.shape[3]
    cw, nw, bs, lam, bv = _params(params)
    M, W = lam.shape[1], cw.shape[3]
    if tuple(k.shape) != (B, N, H, R) or tuple(v.shape[:3]) != (B, N, H):
        raise ValueError("shape mismatch between q, k and v")
    if out is None:
        out = torch.empty((B, N, H, d), dtype=q.dtype).pin_memory()
    if out.is_cuda or not out.is_contiguous() or out.dtype != q.dtype or out.numel() != B * N * H * d:
        raise ValueError("out must be a contiguous CPU tensor of q's dtype with B*N*H*d elements")
    S = ida_state_floats(d, R, M, W)
    if final_state is True:
        final_state = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    elif final_state is False:
        final_state = None
    for name, t in (("final_state", final_state), ("state_in", state_in)):
        if t is not None and (t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32
                              or t.numel() < B * H * S):
            raise ValueError(f"{name} must be a contiguous float32 CPU tensor with B*H*ida_state_floats elements")
    if staging is None:
        nbytes = ida_forward_host_staging_bytes(B, H, N, d, R, M, dt, W, flags)
        staging = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=cw.device)
    if not staging.is_cuda:
        raise ValueError("staging must be a CUDA tensor")
    st = load().ida_forward_host(_p(q), _p(k), _p(v), _p(cw), _p(nw), _p(bs), _p(lam), _p(bv), _p(state_in),
                                 _p(out), _p(final_state), B, H, N, d, R, M, dt, W, int(flags), _p(staging),
                                 staging.numel() * staging.element_size(), _stream_handle(stream))
    _check(st, "ida_forward_host")
    return out, final_state


def ida_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, params: dict,
                out: torch.Tensor | None = None, final_state: torch.Tensor | bool | None = None,
                flags: int = 0, stream=None, workspace: torch.Tensor | None = None,
                state_in: torch.Tensor | None = None):
    """Prefill.  q, k [B,N,H,R], v [B,N,H,d] CUDA tensors (fp32/bf16, contiguous).

    ``params``: dict of float32 CUDA tensors conv_w [2,H,R,W], norm_w/bias
    [H,R+d], lambda/Bvec [H,M,2].  ``final_state``: a [B,H,S] float32 tensor to
    fill, True to allocate one, or None.  ``workspace``: optional CUDA tensor
    (any dtype) handed to ``ida_forward_ws``.  ``state_in``: optional [B,H,S]
    float32 CUDA tensor, the state before position 0 (``ida_forward_from``).
    Returns (out, final_state).
    """
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype")
    B, N, H, R = q.shape
    d = v.shape[3]
    cw, nw, bs, lam, bv = _params(params)
    M, W = lam.shape[1], cw.shape[3]
    if tuple(k.shape) != (B, N, H, R) or tuple(v.shape[:3]) != (B, N, H):
        raise ValueError("shape mismatch between q, k and v")
    if out is None:
        out = torch.empty((B, N, H, d), dtype=q.dtype, device=q.device)
    S = ida_state_floats(d, R, M, W)
    if final_state is True:
        final_state = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    elif final_state is False:
        final_state = None
    if final_state is not None and (final_state.dtype != torch.float32 or final_state.numel() < B * H * S):
        raise ValueError("final_state must be float32 with B*H*ida_state_floats elements")
    if state_in is not None:
        if not (state_in.is_cuda and state_in.is_contiguous() and state_in.dtype == torch.float32
                and state_in.numel() >= B * H * S):
            raise ValueError("state_in must be a contiguous float32 CUDA tensor with B*H*ida_state_floats elements")
        wp, nbytes = None, 0
        if workspace is not None:
            if not workspace.is_cuda:
                raise ValueError("workspace must be a CUDA tensor")
            wp, nbytes = workspace, workspace.numel() * workspace.element_size()
        st = load().ida_forward_from(_p(q), _p(k), _p(v), _p(cw), _p(nw), _p(bs), _p(lam), _p(bv),
                                     _p(state_in), _p(out), _p(final_state), B, H, N, d, R, M, dt, W,
                                     int(flags), _p(wp), nbytes, _stream_handle(stream))
        _check(st, "ida_forward_from")
    elif workspace is None:
        st = load().ida_forward(_p(q), _p(k), _p(v), _p(cw), _p(nw), _p(bs), _p(lam), _p(bv), _p(out),
                                _p(final_state), B, H, N, d, R, M, dt, W, int(flags),
                                _stream_handle(stream))
        _check(st, "ida_forward")
    else:
        if not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        nbytes = workspace.numel() * workspace.element_size()
        st = load().ida_forward_ws(_p(q), _p(k), _p(v), _p(cw), _p(nw), _p(bs), _p(lam), _p(bv),
                                   _p(out), _p(final_state), B, H, N, d, R, M, dt, W, int(flags),
                                   _p(workspace), nbytes, _stream_handle(stream))
        _check(st, "ida_forward_ws")
    return out, final_state


def ida_forward_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, params: dict,
                        out: torch.Tensor, final_state: torch.Tensor | None = None, flags: int = 0,
                        stream=None):
    """Prefill through ``ida_forward_noalloc``: for callers that may not allocate device
    memory, so ``out`` (and ``final_state``, if wanted) must be passed in; the scratch is
    the library's static device array.  Marshalling only, like ``ida_forward``."""
    for t in (q, k, v, out):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("q, k, v and out must be contiguous CUDA tensors")
    dt = _dtype_code(q)
    B, N, H, R = q.shape
    d = v.shape[3]
    cw, nw, bs, lam, bv = _params(params)
    M, W = lam.shape[1], cw.shape[3]
    st = load().ida_forward_noalloc(_p(q), _p(k), _p(v), _p(cw), _p(nw), _p(bs), _p(lam), _p(bv),
                                    _p(out), _p(final_state), B, H, N, d, R, M, dt, W, int(flags),
                                    _stream_handle(stream))
    _check(st, "ida_forward_noalloc")
    return out, final_state


def forward_workspace(q: torch.Tensor, v: torch.Tensor, params: dict, flags: int = 0):
    """A device workspace sized by ``ida_forward_workspace_bytes`` (None when none applies)."""
    B, N, H, R = q.shape
    d = v.shape[3]
    M, W = params["lambda"].shape[1], params["conv_w"].shape[3]
    n = ida_forward_workspace_bytes(B, H, N, d, R, M, _dtype_code(q), W, flags)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=q.device)


def ida_decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, params: dict,
                    state: torch.Tensor, out: torch.Tensor | None = None, flags: int = 0,
                    stream=None) -> torch.Tensor:
    """One decode step.  q, k [B,H,R], v [B,H,d]; ``state`` [B,H,S] float32 updated in place."""
    for t in (q, k, v, state):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("q, k, v and state must be contiguous CUDA tensors")
    dt = _dtype_code(q)
    B, H, R = q.shape
    d = v.shape[2]
    cw, nw, bs, lam, bv = _params(params)
    M, W = lam.shape[1], cw.shape[3]
    if state.dtype != torch.float32 or state.numel() < B * H * ida_state_floats(d, R, M, W):
        raise ValueError("state must be float32 with B*H*ida_state_floats elements")
    if out is None:
        out = torch.empty((B, H, d), dtype=q.dtype, device=q.device)
    st = load().ida_decode_step(_p(q), _p(k), _p(v), _p(cw), _p(nw), _p(bs), _p(lam), _p(bv),
                                _p(state), _p(out), B, H, d, R, M, dt, W, int(flags),
                                _stream_handle(stream))
    _check(st, "ida_decode_step")
    return out


def ida_backward_workspace_bytes(B: int, H: int, N: int, d: int, R: int, M: int, dtype: int,
                                 W: int, flags: int = 0) -> int:
    return int(load().ida_backward_workspace_bytes(B, H, N, d, R, M, dtype, W, flags))


def ida_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, params: dict, dout: torch.Tensor,
                 flags: int = 0, workspace: torch.Tensor | None = None, stream=None,
                 grads: dict | None = None) -> dict:
    """Gradients of the prefill.  q, k [B,N,H,R], v and dout [B,N,H,d] CUDA tensors of one
    dtype.  Returns dict q, k, v (input dtype) and conv_w, norm_w, bias, lambda, Bvec
    (float32, the parameters' shapes), written into ``grads`` when given.  ``workspace``: a
    CUDA tensor of at least ``ida_backward_workspace_bytes`` bytes (allocated here when None)."""
    for t in (q, k, v, dout):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("q, k, v and dout must be contiguous CUDA tensors")
    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype or dout.dtype != q.dtype:
        raise TypeError("q, k, v and dout must share a dtype")
    B, N, H, R = q.shape
    d = v.shape[3]
    cw, nw, bs, lam, bv = _params(params)
    M, W = lam.shape[1], cw.shape[3]
    if tuple(dout.shape) != (B, N, H, d):
        raise ValueError("dout must have the shape of out")
    nbytes = ida_backward_workspace_bytes(B, H, N, d, R, M, dt, W, flags)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    g = grads if grads is not None else {
        "q": torch.empty_like(q), "k": torch.empty_like(k), "v": torch.empty_like(v),
        "conv_w": torch.empty_like(cw), "norm_w": torch.empty_like(nw), "bias": torch.empty_like(bs),
        "lambda": torch.empty_like(lam), "Bvec": torch.empty_like(bv)}
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().ida_backward(_p(q), _p(k), _p(v), _p(cw), _p(nw), _p(bs), _p(lam), _p(bv), _p(dout),
                             _p(g["q"]), _p(g["k"]), _p(g["v"]), _p(g["conv_w"]), _p(g["norm_w"]),
                             _p(g["bias"]), _p(g["lambda"]), _p(g["Bvec"]), B, H, N, d, R, M, dt, W,
                             int(flags), _p(workspace), wbytes, _stream_handle(stream))
    _check(st, "ida_backward")
    return g


def ida_forward_ideal(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, omega: torch.Tensor, params: dict,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The ideal layer on random Fourier features.  q, k [B,N,H,R_in], v [B,N,H,d] CUDA
    tensors of one dtype; omega [H,D,R_in] float32 CUDA; ``params`` as for ida_forward (only
    lambda and Bvec are read).  Returns out [B,N,H,d]."""
    for t in (q, k, v, omega):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("q, k, v and omega must be contiguous CUDA tensors")
    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype")
    if omega.dtype != torch.float32:
        raise TypeError("omega must be float32")
    B, N, H, Rin = q.shape
    d = v.shape[3]
    D = omega.shape[1]
    lam, bv = params["lambda"], params["Bvec"]
    M = lam.shape[1]
    if out is None:
        out = torch.empty((B, N, H, d), dtype=q.dtype, device=q.device)
    st = load().ida_forward_ideal(_p(q), _p(k), _p(v), _p(omega), _p(lam), _p(bv), _p(out), B, H, N, d, Rin, D, M,
                                  dt, _stream_handle(stream))
    _check(st, "ida_forward_ideal")
    return out


def ida_rope(q: torch.Tensor, k: torch.Tensor | None = None, pos0: int = 0, base: float = 10000.0,
             stream=None) -> None:
    """Rotary position embeddings on q (and k) [B,N,H,R] CUDA tensors, in place: channel
    pairs (2i, 2i+1) of the row at position pos0 + t rotate by (pos0 + t) * base^(-2i/R)."""
    for t in (q, k):
        if t is not None and not (t.is_cuda and t.is_contiguous()):
            raise ValueError("q and k must be contiguous CUDA tensors")
    if k is not None and (k.shape != q.shape or k.dtype != q.dtype):
        raise ValueError("k must match q in shape and dtype")
    B, N, H, R = q.shape
    st = load().ida_rope(_p(q), _p(k), B, N, H, R, int(pos0), float(base), _dtype_code(q), _stream_handle(stream))
    _check(st, "ida_rope")


def ida_selftest_bounded_wait(limit_cycles: int, stream=None) -> None:
    """Launch the library's bounded-wait self-test (a wait that runs out on purpose)."""
    _check(load().ida_selftest_bounded_wait(int(limit_cycles), _stream_handle(stream)),
           "ida_selftest_bounded_wait")


def params_to_device(p: dict, device="cuda") -> dict:
    """float32 parameter arrays (e.g. from ``inputs.make_params``) as CUDA tensors."""
    keys = ("conv_w", "norm_w", "bias", "lambda", "Bvec")
    return {k: torch.as_tensor(p[k], dtype=torch.float32).contiguous().to(device) for k in keys}
