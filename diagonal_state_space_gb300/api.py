"""Thin torch binding of libs5.so: the same entry points as include/s5.h.

Argument marshalling only.  Every tensor must already be on the GPU with the
documented dtype, contiguous and 16-byte aligned; nothing is converted or
copied here, and every numeric step runs in the library's kernels.  Complex
arrays are torch.complex64 tensors (interleaved re/im float32, as the C ABI
expects).  Work is queued on the current torch CUDA stream unless ``stream``
is given.
"""
from __future__ import annotations

import torch

from . import _native
from ._native import S5_BF16, S5_F32, S5Error, check

_DT = {torch.float32: S5_F32, torch.bfloat16: S5_BF16}
_DT_NAME = {"f32": S5_F32, "bf16": S5_BF16, torch.float32: S5_F32, torch.bfloat16: S5_BF16}


def _ptr(t, name, dtype=None, shape=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError("%s is required" % name)
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream if isinstance(s, torch.cuda.Stream) else int(s)


def s5_workspace_size(B: int, L: int, H: int, P: int) -> int:
    return int(_native.lib().s5_workspace_size(B, L, H, P))


def new_workspace(B: int, L: int, H: int, P: int, device=None) -> torch.Tensor:
    """A zero-filled workspace for s5_forward / s5_forward_varying_dt (the
    caller's allocation, made here with torch for convenience)."""
    n = s5_workspace_size(B, L, H, P)
    if n == 0:
        raise ValueError("invalid sizes for a workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def s5_discretize(lam, log_dt, b_tilde, lambda_bar=None, b_bar=None, stream=None):
    """Zero-order hold; returns (lambda_bar [P] complex64, b_bar [P,H] complex64)."""
    P, H = b_tilde.shape
    if lambda_bar is None:
        lambda_bar = torch.empty(P, dtype=torch.complex64, device=b_tilde.device)
    if b_bar is None:
        b_bar = torch.empty(P, H, dtype=torch.complex64, device=b_tilde.device)
    c64 = torch.complex64
    code = _native.lib().s5_discretize(
        _ptr(lam, "lambda", c64, (P,)), _ptr(log_dt, "log_dt", torch.float32, (P,)),
        _ptr(b_tilde, "b_tilde", c64), P, H, _ptr(lambda_bar, "lambda_bar", c64, (P,)),
        _ptr(b_bar, "b_bar", c64, (P, H)), _stream(stream))
    check("s5_discretize", code)
    return lambda_bar, b_bar


_METHOD = {"zoh": 0, "bilinear": 1}


def s5_discretize_ex(lam, log_dt, b_tilde, method="zoh", clip_re=0.0, dt_scale=1.0, lambda_bar=None,
                     b_bar=None, stream=None):
    """Discretisation with options: method "zoh" or "bilinear", clip_eigs
    threshold clip_re (0 = none; the official value is -1e-4), sampling-rate
    factor dt_scale = old rate / new rate.  Returns (lambda_bar, b_bar)."""
    P, H = b_tilde.shape
    if lambda_bar is None:
        lambda_bar = torch.empty(P, dtype=torch.complex64, device=b_tilde.device)
    if b_bar is None:
        b_bar = torch.empty(P, H, dtype=torch.complex64, device=b_tilde.device)
    c64 = torch.complex64
    code = _native.lib().s5_discretize_ex(
        _ptr(lam, "lambda", c64, (P,)), _ptr(log_dt, "log_dt", torch.float32, (P,)),
        _ptr(b_tilde, "b_tilde", c64), P, H, _METHOD[method], float(clip_re), float(dt_scale),
        _ptr(lambda_bar, "lambda_bar", c64, (P,)), _ptr(b_bar, "b_bar", c64, (P, H)), _stream(stream))
    check("s5_discretize_ex", code)
    return lambda_bar, b_bar


def s5_step(lambda_bar, b_bar, c_tilde, d, x, u, y=None, stream=None):
    """One streaming step: x [B,P] complex64 is updated in place; returns y [B,H]."""
    P, H = b_bar.shape
    Bn = u.shape[0]
    if y is None:
        y = torch.empty(Bn, H, dtype=torch.float32, device=u.device)
    c64 = torch.complex64
    code = _native.lib().s5_step(
        _ptr(lambda_bar, "lambda_bar", c64, (P,)), _ptr(b_bar, "b_bar", c64, (P, H)),
        _ptr(c_tilde, "c_tilde", c64, (H, P)), _ptr(d, "d", torch.float32, (H,)),
        _ptr(x, "x", c64, (Bn, P)), _ptr(u, "u", torch.float32, (Bn, H)),
        _ptr(y, "y", torch.float32, (Bn, H)), Bn, H, P, _stream(stream))
    check("s5_step", code)
    return y


def s5_bidirectional_workspace_size(B, L, H, P, u_dtype=torch.float32, y_dtype=None) -> int:
    y_dtype = u_dtype if y_dtype is None else y_dtype
    return int(_native.lib().s5_bidirectional_workspace_size(B, L, H, P, _DT[u_dtype], _DT[y_dtype]))


def s5_forward_bidirectional(lambda_bar, b_bar, c_tilde2, d, u, y=None, y_dtype=None, proj_dtype="f32",
                             workspace=None, stream=None):
    """Bidirectional S5 layer: c_tilde2 [H,2P] holds the forward modes' C~ in
    columns 0..P-1 and the backward modes' in P..2P-1.  Returns y."""
    P = b_bar.shape[0]
    Bn, L, H = u.shape
    if u.dtype not in _DT:
        raise ValueError("u must be float32 or bfloat16")
    ydt = u.dtype if y_dtype is None else y_dtype
    if isinstance(ydt, str):
        ydt = {"f32": torch.float32, "bf16": torch.bfloat16}[ydt]
    if y is None:
        y = torch.empty(Bn, L, H, dtype=ydt, device=u.device)
    if workspace is None:
        n = s5_bidirectional_workspace_size(Bn, L, H, P, u.dtype, y.dtype)
        if n == 0:
            raise ValueError("invalid sizes for a workspace")
        workspace = torch.zeros(n, dtype=torch.uint8, device=u.device)
    c64 = torch.complex64
    code = _native.lib().s5_forward_bidirectional(
        _ptr(lambda_bar, "lambda_bar", c64, (P,)), _ptr(b_bar, "b_bar", c64, (P, H)),
        _ptr(c_tilde2, "c_tilde2", c64, (H, 2 * P)), _ptr(d, "d", torch.float32, (H,)),
        _ptr(u, "u"), _DT[u.dtype], _ptr(y, "y", None, (Bn, L, H)), _DT[y.dtype], _DT_NAME[proj_dtype],
        Bn, L, H, P, _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    check("s5_forward_bidirectional", code)
    return y


def _fwd_common(u, y, y_dtype, proj_dtype, x0, x_last, workspace, P):
    Bn, L, H = u.shape
    if u.dtype not in _DT:
        raise ValueError("u must be float32 or bfloat16")
    ydt = u.dtype if y_dtype is None else y_dtype
    if isinstance(ydt, str):
        ydt = {"f32": torch.float32, "bf16": torch.bfloat16}[ydt]
    if y is None:
        y = torch.empty(Bn, L, H, dtype=ydt, device=u.device)
    if x_last is True:
        x_last = torch.empty(Bn, P, dtype=torch.complex64, device=u.device)
    if workspace is None:
        workspace = new_workspace(Bn, L, H, P, u.device)
    return Bn, L, H, y, x_last, workspace, _DT_NAME[proj_dtype]


def s5_forward(lambda_bar, b_bar, c_tilde, d, u, y=None, y_dtype=None, proj_dtype="f32",
               x0=None, x_last=None, workspace=None, stream=None):
    """Time-invariant S5 forward.  Returns y, or (y, x_last) when x_last is a
    tensor or True."""
    P = b_bar.shape[0]
    Bn, L, H, y, x_last, ws, pd = _fwd_common(u, y, y_dtype, proj_dtype, x0, x_last, workspace, P)
    c64 = torch.complex64
    code = _native.lib().s5_forward(
        _ptr(lambda_bar, "lambda_bar", c64, (P,)), _ptr(b_bar, "b_bar", c64, (P, H)),
        _ptr(c_tilde, "c_tilde", c64, (H, P)), _ptr(d, "d", torch.float32, (H,)),
        _ptr(u, "u"), _DT[u.dtype], _ptr(y, "y", None, (Bn, L, H)), _DT[y.dtype], pd,
        Bn, L, H, P, _ptr(x0, "x0", c64, (Bn, P), True),
        _ptr(x_last, "x_last", c64, (Bn, P), True), _ptr(ws, "workspace", torch.uint8),
        ws.numel(), _stream(stream))
    check("s5_forward", code)
    return y if x_last is None else (y, x_last)


def s5_forward_varying_dt(lam, log_dt, b_tilde, c_tilde, d, dt_scale, u, y=None, y_dtype=None,
                          proj_dtype="f32", x0=None, x_last=None, workspace=None, stream=None):
    """Irregular-sampling S5 forward (interval dt_scale[b,k]*exp(log_dt[n]))."""
    P = b_tilde.shape[0]
    Bn, L, H, y, x_last, ws, pd = _fwd_common(u, y, y_dtype, proj_dtype, x0, x_last, workspace, P)
    c64 = torch.complex64
    code = _native.lib().s5_forward_varying_dt(
        _ptr(lam, "lambda", c64, (P,)), _ptr(log_dt, "log_dt", torch.float32, (P,)),
        _ptr(b_tilde, "b_tilde", c64, (P, H)), _ptr(c_tilde, "c_tilde", c64, (H, P)),
        _ptr(d, "d", torch.float32, (H,)), _ptr(dt_scale, "dt_scale", torch.float32, (Bn, L)),
        _ptr(u, "u"), _DT[u.dtype], _ptr(y, "y", None, (Bn, L, H)), _DT[y.dtype], pd,
        Bn, L, H, P, _ptr(x0, "x0", c64, (Bn, P), True),
        _ptr(x_last, "x_last", c64, (Bn, P), True), _ptr(ws, "workspace", torch.uint8),
        ws.numel(), _stream(stream))
    check("s5_forward_varying_dt", code)
    return y if x_last is None else (y, x_last)


def s5_forward_noalloc(lambda_bar, b_bar, c_tilde, d, u, y, proj_dtype="f32", x0=None,
                       x_last=None, stream=None):
    """s5_forward for callers that cannot allocate device memory: no workspace,
    and no tensor is created here either (y, and x_last if wanted, are the
    caller's).  The library keeps the carry scratch in a fixed device array of
    S5_NOALLOC_SCRATCH_BYTES; larger problems are rejected.  Calls that overlap
    on the GPU share that array and race, so serialize them."""
    P = b_bar.shape[0]
    Bn, L, H = u.shape
    need = s5_workspace_size(Bn, L, H, P)
    if need > _native.S5_NOALLOC_SCRATCH_BYTES:
        raise S5Error("s5_forward_noalloc", 1,
                      "needs %d bytes of carry scratch, more than the library's fixed %d"
                      % (need, _native.S5_NOALLOC_SCRATCH_BYTES))
    c64 = torch.complex64
    code = _native.lib().s5_forward_noalloc(
        _ptr(lambda_bar, "lambda_bar", c64, (P,)), _ptr(b_bar, "b_bar", c64, (P, H)),
        _ptr(c_tilde, "c_tilde", c64, (H, P)), _ptr(d, "d", torch.float32, (H,)),
        _ptr(u, "u"), _DT[u.dtype], _ptr(y, "y", None, (Bn, L, H)), _DT[y.dtype],
        _DT_NAME[proj_dtype], Bn, L, H, P, _ptr(x0, "x0", c64, (Bn, P), True),
        _ptr(x_last, "x_last", c64, (Bn, P), True), _stream(stream))
    check("s5_forward_noalloc", code)
    return y if x_last is None else (y, x_last)


def s5_sync_status(workspace, stream=None) -> int:
    """Waits for the stream; returns and clears the latched device status."""
    return int(_native.lib().s5_sync_status(_ptr(workspace, "workspace", torch.uint8),
                                            _stream(stream)))


__all__ = ["s5_discretize", "s5_discretize_ex", "s5_forward", "s5_forward_varying_dt",
           "s5_forward_bidirectional", "s5_step", "s5_forward_noalloc", "s5_workspace_size",
           "s5_bidirectional_workspace_size", "s5_sync_status", "new_workspace", "S5Error", "S5_F32",
           "S5_BF16"]
