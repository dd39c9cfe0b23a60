"""Helpers of the GPU parity tests: seeded inputs to the device, the oracle on
the same stored values, and the error measures."""
import os

import numpy as np
import torch

import oracle
from diagonal_state_space_gb300 import api


def _pair(got, ref):
    cplx = np.iscomplexobj(got) or np.iscomplexobj(ref)
    dt = np.complex128 if cplx else np.float64
    return np.asarray(got, dt), np.asarray(ref, dt)


def rel_l2(got, ref):
    got, ref = _pair(got, ref)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def max_abs(got, ref):
    got, ref = _pair(got, ref)
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


# (test, quantity, rel-L2, max-abs, max |ref|, tolerance) of every check made
# in this session; conftest prints them as the parity table.
PARITY_LOG = []


def check(got, ref, tol, what="y"):
    """Asserts rel-L2(got, ref) <= tol; the message and the parity table give
    the max-abs error beside it."""
    got, ref = _pair(got, ref)
    r, m = rel_l2(got, ref), max_abs(got, ref)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    PARITY_LOG.append((test, what, r, m, scale, tol))
    assert r <= tol, "%s: rel-L2 %.3e > %.1e (max-abs %.3e, max |ref| %.3e)" % (what, r, tol, m, scale)
    return r, m


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def layer_to_device(inp, u_dtype="f32"):
    return dict(
        u=dev(inp["u"], torch.bfloat16 if u_dtype == "bf16" else torch.float32),
        lam=dev(inp["lambda_"]), log_dt=dev(inp["log_dt"]), b_tilde=dev(inp["b_tilde"]),
        c_tilde=dev(inp["c_tilde"]), d=dev(inp["d"]),
        g=dev(inp["g"]) if "g" in inp else None)


def oracle_forward(inp, x0=None, seqs=None, c64_params=False):
    """Oracle y and x_last for the time-invariant layer (optionally only for
    the listed sequences).  With c64_params the oracle's own lambda_bar and
    B_bar are first rounded to complex64, the type the C ABI stores them in:
    a state carried from x0 over L steps picks up about L ulps of lambda_bar's
    rounding (a relative 2e-5 at L = 1024), which the float64 oracle does not
    have; the rounded oracle isolates the kernel's own arithmetic error."""
    lb, bb = oracle.discretize(inp["lambda_"], inp["log_dt"], inp["b_tilde"])
    if c64_params:
        lb = lb.astype(np.complex64).astype(np.complex128)
        bb = bb.astype(np.complex64).astype(np.complex128)
    u = inp["u"] if seqs is None else inp["u"][seqs]
    x0s = None if x0 is None else (x0 if seqs is None else x0[seqs])
    return oracle.forward(lb, bb, inp["c_tilde"], inp["d"], u, x0=x0s)


def oracle_forward_varying(inp, x0=None, seqs=None):
    u = inp["u"] if seqs is None else inp["u"][seqs]
    g = inp["g"] if seqs is None else inp["g"][seqs]
    x0s = None if x0 is None else (x0 if seqs is None else x0[seqs])
    return oracle.forward_varying_dt(inp["lambda_"], inp["log_dt"], inp["b_tilde"],
                                     inp["c_tilde"], inp["d"], g, u, x0=x0s)


def gpu_forward(t, u_dtype="f32", y_dtype=None, proj_dtype="f32", x0=None, want_x_last=False,
                workspace=None):
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    out = api.s5_forward(lb, bb, t["c_tilde"], t["d"], t["u"], y_dtype=y_dtype,
                         proj_dtype=proj_dtype, x0=x0, x_last=True if want_x_last else None,
                         workspace=workspace)
    return out


def gpu_forward_varying(t, y_dtype=None, proj_dtype="f32", x0=None, want_x_last=False,
                        workspace=None):
    return api.s5_forward_varying_dt(t["lam"], t["log_dt"], t["b_tilde"], t["c_tilde"], t["d"],
                                     t["g"], t["u"], y_dtype=y_dtype, proj_dtype=proj_dtype,
                                     x0=x0, x_last=True if want_x_last else None,
                                     workspace=workspace)


def host(t):
    if t.dtype == torch.complex64:
        return t.cpu().numpy().astype(np.complex128)
    return t.float().cpu().numpy().astype(np.float64)
