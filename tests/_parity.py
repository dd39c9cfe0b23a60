"""Helpers of the GPU parity tests: seeded inputs to the device, the oracle on
the same stored values, and the error measures."""
import numpy as np
import torch

import oracle
from diagonal_state_space_gb300 import api


def rel_l2(got, ref):
    cplx = np.iscomplexobj(got) or np.iscomplexobj(ref)
    dt = np.complex128 if cplx else np.float64
    got = np.asarray(got, dt)
    ref = np.asarray(ref, dt)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def layer_to_device(inp, u_dtype="f32"):
    return dict(
        u=dev(inp["u"], torch.bfloat16 if u_dtype == "bf16" else torch.float32),
        lam=dev(inp["lambda_"]), log_dt=dev(inp["log_dt"]), b_tilde=dev(inp["b_tilde"]),
        c_tilde=dev(inp["c_tilde"]), d=dev(inp["d"]),
        g=dev(inp["g"]) if "g" in inp else None)


def oracle_forward(inp, x0=None, seqs=None):
    """Oracle y and x_last for the time-invariant layer (optionally only for
    the listed sequences)."""
    lb, bb = oracle.discretize(inp["lambda_"], inp["log_dt"], inp["b_tilde"])
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
