"""Float64 CPU oracle for the S5 layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
nothing here imports the product package.

The arithmetic lives in ``s5_oracle.c`` (plain C99, ``double`` and
``double complex``, single-threaded, sequential recurrence); this module only
compiles it with gcc and marshals numpy arrays.  Every input is promoted to
float64 / complex128 before the call, so the oracle sees exactly the stored
values the GPU path sees.

Pinned by ``tests/test_oracle_pins.py`` against closed forms, a brute-force
associative scan, an ODE integrator, the worked example of the S4 page and
finite differences.  Parity unpinned: nothing (every exported function has at
least one pin).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "s5_oracle.c")
_LIB = os.path.join(_HERE, "libs5_oracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no -march, no fast-math). Returns the .so path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = ctypes.CDLL(_LIB)
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _c128(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.complex128))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


_I = ctypes.c_int


def discretize(lam, log_dt, b_tilde):
    """Zero-order hold: (lambda [P], log_dt [P], B~ [P,H]) -> (lambda_bar [P], B_bar [P,H])."""
    lam, log_dt, b_tilde = _c128(lam), _f64(log_dt), _c128(b_tilde)
    P, H = b_tilde.shape
    lb = np.empty(P, np.complex128)
    bb = np.empty((P, H), np.complex128)
    _load().s5o_discretize(_I(P), _I(H), _p(lam), _p(log_dt), _p(b_tilde), _p(lb), _p(bb))
    return lb, bb


def discretize_ex(lam, log_dt, b_tilde, method="zoh", clip_re=0.0, dt_scale=1.0):
    """Discretisation with options: method "zoh" or "bilinear", clip_eigs
    threshold clip_re (0 = none; the official value is -1e-4), and the
    sampling-rate rescaling factor dt_scale = old rate / new rate."""
    lam, log_dt, b_tilde = _c128(lam), _f64(log_dt), _c128(b_tilde)
    P, H = b_tilde.shape
    lb = np.empty(P, np.complex128)
    bb = np.empty((P, H), np.complex128)
    m = {"zoh": 0, "bilinear": 1}[method]
    _load().s5o_discretize_ex(_I(P), _I(H), _p(lam), _p(log_dt), _p(b_tilde), _I(m),
                              ctypes.c_double(clip_re), ctypes.c_double(dt_scale), _p(lb), _p(bb))
    return lb, bb


def step(lambda_bar, b_bar, c_tilde, d, x, u):
    """One streaming step: returns (x_new [B,P], y [B,H]) for x [B,P], u [B,H]."""
    lb, bb, ct, d = _c128(lambda_bar), _c128(b_bar), _c128(c_tilde), _f64(d)
    x = _c128(x).copy()
    u = _f64(u)
    Bn, H = u.shape
    P = lb.shape[0]
    y = np.empty((Bn, H), np.float64)
    _load().s5o_step(_I(Bn), _I(H), _I(P), _p(lb), _p(bb), _p(ct), _p(d), _p(x), _p(u), _p(y))
    return x, y


def forward_bidirectional(lambda_bar, b_bar, c_tilde2, d, u):
    """Bidirectional layer over u [B,L,H] with C~ [H,2P] (forward modes, then
    backward modes); returns y [B,L,H]."""
    lb, bb, ct, d, u = _c128(lambda_bar), _c128(b_bar), _c128(c_tilde2), _f64(d), _f64(u)
    Bn, L, H = u.shape
    P = lb.shape[0]
    assert ct.shape == (H, 2 * P)
    y = np.empty((Bn, L, H), np.float64)
    _load().s5o_forward_bidirectional(_I(Bn), _I(L), _I(H), _I(P), _p(lb), _p(bb), _p(ct), _p(d),
                                      _p(u), _p(y))
    return y


def forward(lambda_bar, b_bar, c_tilde, d, u, x0=None, return_states=False):
    """Time-invariant layer over u [B,L,H]; returns y [B,L,H] and x_last [B,P]
    (or all states [B,L,P] when ``return_states``)."""
    lb, bb, ct, d, u = _c128(lambda_bar), _c128(b_bar), _c128(c_tilde), _f64(d), _f64(u)
    Bn, L, H = u.shape
    P = lb.shape[0]
    assert bb.shape == (P, H) and ct.shape == (H, P) and d.shape == (H,)
    x0 = None if x0 is None else _c128(x0).reshape(Bn, P)
    y = np.empty((Bn, L, H), np.float64)
    lib = _load()
    if return_states:
        st = np.empty((Bn, L, P), np.complex128)
        lib.s5o_forward_states(_I(Bn), _I(L), _I(H), _I(P), _p(lb), _p(bb), _p(ct), _p(d),
                               _p(u), _p(x0), _p(y), _p(st))
        return y, st
    xl = np.empty((Bn, P), np.complex128)
    lib.s5o_forward(_I(Bn), _I(L), _I(H), _I(P), _p(lb), _p(bb), _p(ct), _p(d), _p(u),
                    _p(x0), _p(y), _p(xl))
    return y, xl


def forward_varying_dt(lam, log_dt, b_tilde, c_tilde, d, g, u, x0=None):
    """Irregular sampling: interval g[b,k]*exp(log_dt[n]) at step k, mode n."""
    lam, log_dt, bt, ct = _c128(lam), _f64(log_dt), _c128(b_tilde), _c128(c_tilde)
    d, g, u = _f64(d), _f64(g), _f64(u)
    Bn, L, H = u.shape
    P = lam.shape[0]
    assert g.shape == (Bn, L)
    x0 = None if x0 is None else _c128(x0).reshape(Bn, P)
    y = np.empty((Bn, L, H), np.float64)
    xl = np.empty((Bn, P), np.complex128)
    _load().s5o_forward_varying_dt(_I(Bn), _I(L), _I(H), _I(P), _p(lam), _p(log_dt), _p(bt),
                                   _p(ct), _p(d), _p(g), _p(u), _p(x0), _p(y), _p(xl))
    return y, xl


def layernorm(x):
    x = _f64(x)
    H = x.shape[-1]
    z = np.empty_like(x)
    _load().s5o_layernorm(ctypes.c_size_t(x.size // H), _I(H), _p(x), _p(z))
    return z


def gate(y, W):
    y, W = _f64(y), _f64(W)
    H = y.shape[-1]
    out = np.empty_like(y)
    _load().s5o_gate(ctypes.c_size_t(y.size // H), _I(H), _p(y), _p(W), _p(out))
    return out


def stack(params, u0, G=None):
    """Layer stack forward (and backward when G is given).

    params: dict of per-layer stacked arrays lambda [nl,P], log_dt [nl,P],
    b_tilde [nl,P,H], c_tilde [nl,H,P], d [nl,H], W [nl,H,H].
    Returns u_out, or (u_out, grads) with grads keys
    du0, dlambda, dlog_dt, db_tilde, dc_tilde, dd, dW.
    """
    lam, log_dt = _c128(params["lambda"]), _f64(params["log_dt"])
    bt, ct = _c128(params["b_tilde"]), _c128(params["c_tilde"])
    d, W, u0 = _f64(params["d"]), _f64(params["W"]), _f64(u0)
    nl, P = lam.shape
    Bn, L, H = u0.shape
    u_out = np.empty_like(u0)
    lib = _load()
    if G is None:
        lib.s5o_stack(_I(nl), _I(Bn), _I(L), _I(H), _I(P), _p(lam), _p(log_dt), _p(bt), _p(ct),
                      _p(d), _p(W), _p(u0), _p(u_out), None, None, None, None, None, None,
                      None, None)
        return u_out
    G = _f64(G)
    gr = dict(du0=np.empty_like(u0), dlambda=np.empty_like(lam), dlog_dt=np.empty_like(log_dt),
              db_tilde=np.empty_like(bt), dc_tilde=np.empty_like(ct), dd=np.empty_like(d),
              dW=np.empty_like(W))
    lib.s5o_stack(_I(nl), _I(Bn), _I(L), _I(H), _I(P), _p(lam), _p(log_dt), _p(bt), _p(ct),
                  _p(d), _p(W), _p(u0), _p(u_out), _p(G), _p(gr["du0"]), _p(gr["dlambda"]),
                  _p(gr["dlog_dt"]), _p(gr["db_tilde"]), _p(gr["dc_tilde"]), _p(gr["dd"]),
                  _p(gr["dW"]))
    return u_out, gr
