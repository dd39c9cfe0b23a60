"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs.

Bars (written here, applied per output tensor): relative L2 error <= 1e-5 for
the float32 paths and <= 2e-2 where projections or outputs are bfloat16.
Because D*u dominates ||y|| under these generators, every float32 case is
also run with D = 0 so that the bar applies to the SSM term itself.
"""
import numpy as np
import pytest
import torch

from diagonal_state_space_gb300 import api
from diagonal_state_space_gb300.workloads import WORKLOADS, make_inputs, make_layer_inputs

from _parity import (dev, gpu_forward, gpu_forward_varying, host, layer_to_device,
                     oracle_forward, oracle_forward_varying, check)
import oracle

pytestmark = pytest.mark.gpu

FP32_TOL = 1e-5
BF16_TOL = 2e-2


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    torch.cuda.init()


def _zero_d(inp):
    out = dict(inp)
    out["d"] = np.zeros_like(inp["d"])
    return out


# --------------------------------------------------------------------------
# a1: discretisation
# --------------------------------------------------------------------------
@pytest.mark.parametrize("P,H", [(1, 1), (32, 32), (64, 128), (128, 256), (300, 7)])
def test_discretize_matches_oracle(P, H):
    inp = make_layer_inputs(1, 1, H, P, seed=5 + P)
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    olb, obb = oracle.discretize(inp["lambda_"], inp["log_dt"], inp["b_tilde"])
    assert np.max(np.abs(host(lb) - olb) / np.abs(olb)) < 2e-7
    assert np.max(np.abs(host(bb) - obb)) <= 2e-7 * np.max(np.abs(obb)) + 1e-30
    np.testing.assert_allclose(host(bb), obb, rtol=3e-7, atol=1e-12)


def test_discretize_large_phases_and_options():
    """Modes whose phase Im(lambda)*Delta runs to ~120 rad, strongly damped
    modes, and every option path, against the float64 oracle at the same
    bars (lambda_bar 2e-7 relative per element, B_bar 3e-7)."""
    rng = np.random.default_rng(21)
    n = np.arange(128)
    lam = np.concatenate([-0.5 + 1j * np.pi * n,
                          rng.normal(0, 3, 128) - 0.1 + 1j * rng.normal(0, 400, 128),
                          -rng.uniform(0.5, 40, 32) + 1j * rng.uniform(-5, 5, 32)]).astype(np.complex64)
    P = lam.shape[0]
    log_dt = rng.uniform(np.log(1e-3), np.log(3e-1), P).astype(np.float32)
    H = 40
    bt = (rng.standard_normal((P, H)) + 1j * rng.standard_normal((P, H))).astype(np.complex64)
    for method, clip_re, dt_scale in [("zoh", 0.0, 1.0), ("bilinear", 0.0, 1.0), ("zoh", -1e-4, 0.37),
                                      ("bilinear", -1e-4, 2.5)]:
        lb, bb = api.s5_discretize_ex(dev(lam), dev(log_dt), dev(bt), method, clip_re, dt_scale)
        # the C ABI takes clip_re and dt_scale as float: the oracle gets the same values
        olb, obb = oracle.discretize_ex(lam, log_dt, bt, method, float(np.float32(clip_re)),
                                        float(np.float32(dt_scale)))
        np.testing.assert_allclose(host(lb), olb, rtol=2e-7, atol=1e-30)
        np.testing.assert_allclose(host(bb), obb, rtol=3e-7, atol=1e-30)


def test_discretize_zero_pole_and_tiny_interval():
    lam = np.array([0.0, -0.5 + 1e-3j, -0.5 + 100j, -1e-6], np.complex64)
    log_dt = np.log(np.array([0.37, 1e-6, 0.1, 1e-3])).astype(np.float32)
    bt = (np.arange(8).reshape(4, 2) + 1j).astype(np.complex64)
    lb, bb = api.s5_discretize(dev(lam), dev(log_dt), dev(bt))
    olb, obb = oracle.discretize(lam, log_dt, bt)
    np.testing.assert_allclose(host(lb), olb, rtol=2e-7, atol=1e-30)
    np.testing.assert_allclose(host(bb), obb, rtol=3e-7, atol=1e-30)
    assert np.all(np.isfinite(host(bb)))


# --------------------------------------------------------------------------
# a2 + a4 + a5: time-invariant forward
# --------------------------------------------------------------------------
SHAPES = [(1, 1, 1, 1), (2, 5, 3, 1), (3, 77, 5, 3), (2, 200, 33, 17), (1, 129, 16, 8),
          (2, 1000, 130, 65), (1, 300, 24, 300), (5, 64, 64, 64), (1, 4097, 32, 32)]


@pytest.mark.parametrize("B,L,H,P", SHAPES)
@pytest.mark.parametrize("zero_d", [False, True])
def test_forward_fp32_ragged_shapes(B, L, H, P, zero_d):
    inp = make_layer_inputs(B, L, H, P, seed=B * 1000 + L + H + P)
    if zero_d:
        inp = _zero_d(inp)
    t = layer_to_device(inp)
    y, xl = gpu_forward(t, want_x_last=True)
    oy, oxl = oracle_forward(inp)
    check(host(y), oy, FP32_TOL, "host(y)")
    check(host(xl), oxl, FP32_TOL, "host(xl)")


@pytest.mark.parametrize("u_dtype,y_dtype,tol", [("f32", "bf16", BF16_TOL), ("bf16", "f32", FP32_TOL),
                                                  ("bf16", "bf16", BF16_TOL)])
def test_forward_storage_dtypes(u_dtype, y_dtype, tol):
    inp = make_layer_inputs(3, 333, 64, 32, seed=77, u_dtype=u_dtype)
    t = layer_to_device(inp, u_dtype)
    y = gpu_forward(t, y_dtype=y_dtype)
    assert y.dtype == (torch.bfloat16 if y_dtype == "bf16" else torch.float32)
    oy, _ = oracle_forward(inp)
    check(host(y), oy, tol, "host(y)")


def test_forward_streaming_in_two_calls():
    """x_last of one call as x0 of the next equals one call over the whole sequence."""
    inp = make_layer_inputs(3, 500, 48, 40, seed=9)
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    u1, u2 = t["u"][:, :203].contiguous(), t["u"][:, 203:].contiguous()
    y1, x1 = api.s5_forward(lb, bb, t["c_tilde"], t["d"], u1, x_last=True)
    y2, x2 = api.s5_forward(lb, bb, t["c_tilde"], t["d"], u2, x0=x1, x_last=True)
    oy, oxl = oracle_forward(inp)
    check(np.concatenate([host(y1), host(y2)], 1), oy, FP32_TOL, "np.concatenate([host(y1), host(y2)], 1)")
    check(host(x2), oxl, FP32_TOL, "host(x2)")
    # and an explicit non-zero x0 against the oracle
    x0 = (np.random.default_rng(3).standard_normal((3, 40)) +
          1j * np.random.default_rng(4).standard_normal((3, 40))).astype(np.complex64)
    y, xl = api.s5_forward(lb, bb, t["c_tilde"], t["d"], t["u"], x0=dev(x0), x_last=True)
    oy, oxl = oracle_forward(inp, x0=x0)
    check(host(y), oy, FP32_TOL, "host(y)")
    check(host(xl), oxl, FP32_TOL, "host(xl)")


def test_forward_empty_inputs():
    inp = make_layer_inputs(2, 1, 8, 4, seed=1)
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    u0 = torch.empty(2, 0, 8, device="cuda")
    x0 = torch.randn(2, 4, dtype=torch.complex64, device="cuda")
    y, xl = api.s5_forward(lb, bb, t["c_tilde"], t["d"], u0, x0=x0, x_last=True)
    assert y.shape == (2, 0, 8)
    assert torch.equal(xl, x0)
    y, xl = api.s5_forward(lb, bb, t["c_tilde"], t["d"], u0, x_last=True)
    assert torch.count_nonzero(xl) == 0
    ub = torch.empty(0, 5, 8, device="cuda")
    assert api.s5_forward(lb, bb, t["c_tilde"], t["d"], ub).shape == (0, 5, 8)


def test_forward_repeat_runs_agree():
    inp = make_layer_inputs(4, 2000, 64, 64, seed=11)
    t = layer_to_device(inp)
    ws = api.new_workspace(4, 2000, 64, 64)
    y1 = gpu_forward(t, workspace=ws)
    y2 = gpu_forward(t, workspace=ws)
    check(host(y1), host(y2), 1e-6, "host(y1)")
    assert api.s5_sync_status(ws) == 0


# --------------------------------------------------------------------------
# a3: irregular sampling
# --------------------------------------------------------------------------
VSHAPES = [(1, 1, 1, 1), (1, 100, 8, 4), (2, 333, 40, 24), (3, 64, 16, 300), (2, 517, 256, 128)]


@pytest.mark.parametrize("B,L,H,P", VSHAPES)
@pytest.mark.parametrize("zero_d", [False, True])
def test_varying_dt_ragged_shapes(B, L, H, P, zero_d):
    inp = make_layer_inputs(B, L, H, P, seed=500 + B + L + H + P, varying_dt=True)
    inp["g"][:, ::7] = 0.0                 # some zero gaps
    if zero_d:
        inp = _zero_d(inp)
    t = layer_to_device(inp)
    y, xl = gpu_forward_varying(t, want_x_last=True)
    oy, oxl = oracle_forward_varying(inp)
    check(host(y), oy, FP32_TOL, "host(y)")
    check(host(xl), oxl, FP32_TOL, "host(xl)")


def test_varying_dt_large_gaps_and_streaming():
    inp = make_layer_inputs(2, 400, 32, 64, seed=8, varying_dt=True)
    inp["g"] *= 10.0                        # phases of several hundred radians
    inp = _zero_d(inp)
    t = layer_to_device(inp)
    y1, x1 = api.s5_forward_varying_dt(t["lam"], t["log_dt"], t["b_tilde"], t["c_tilde"], t["d"],
                                       t["g"][:, :150].contiguous(), t["u"][:, :150].contiguous(),
                                       x_last=True)
    y2 = api.s5_forward_varying_dt(t["lam"], t["log_dt"], t["b_tilde"], t["c_tilde"], t["d"],
                                   t["g"][:, 150:].contiguous(), t["u"][:, 150:].contiguous(),
                                   x0=x1)
    oy, _ = oracle_forward_varying(inp)
    check(np.concatenate([host(y1), host(y2)], 1), oy, FP32_TOL, "np.concatenate([host(y1), host(y2)], 1)")


@pytest.mark.parametrize("bad", [-1.0, float("nan"), float("inf")])
def test_varying_dt_bad_gap_latches_status(bad):
    inp = make_layer_inputs(1, 50, 8, 4, seed=2, varying_dt=True)
    inp["g"][0, 17] = bad
    t = layer_to_device(inp)
    ws = api.new_workspace(1, 50, 8, 4)
    gpu_forward_varying(t, workspace=ws)
    assert api.s5_sync_status(ws) == 5          # S5_ERR_NONFINITE
    assert api.s5_sync_status(ws) == 0          # cleared by the read
    inp["g"][0, 17] = 1.0
    t = layer_to_device(inp)
    y = gpu_forward_varying(t, workspace=ws)
    assert api.s5_sync_status(ws) == 0
    check(host(y), oracle_forward_varying(inp)[0], FP32_TOL, "host(y)")


# --------------------------------------------------------------------------
# Failure detection: a carry flag that nothing sets.  The header word at
# byte 16 names a tile (plus one) whose flags are never published, the word
# at byte 20 sets the wait limit in microseconds.  The waiting tile gives up,
# latches S5_ERR_TIMEOUT and the launch completes; the workspace stays usable.
# --------------------------------------------------------------------------
def test_carry_wait_timeout_is_reported_and_recoverable():
    inp = make_layer_inputs(1, 4096, 32, 32, seed=3)
    t = layer_to_device(inp)
    ws = api.new_workspace(1, 4096, 32, 32)
    words = ws.view(torch.int32)
    words[4] = 1          # tile 0 never publishes
    words[5] = 2000       # 2 ms wait limit
    gpu_forward(t, workspace=ws)
    assert api.s5_sync_status(ws) == 4          # S5_ERR_TIMEOUT
    words[4] = 0
    words[5] = 0
    y = gpu_forward(t, workspace=ws)
    assert api.s5_sync_status(ws) == 0
    check(host(y), oracle_forward(inp)[0], FP32_TOL, "host(y)")


# --------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the benchmark times; the
# oracle computes every sequence (each workload takes it seconds).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["small", "fp32", "pathx_bf16", "irregular"])
@pytest.mark.parametrize("zero_d", [False, True])
def test_full_size_workloads(name, zero_d):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    if zero_d:
        inp = _zero_d(inp)
    t = layer_to_device(inp, w.u_dtype)
    if w.varying_dt:
        y, xl = gpu_forward_varying(t, proj_dtype=w.proj_dtype, want_x_last=True)
    else:
        y, xl = gpu_forward(t, u_dtype=w.u_dtype, proj_dtype=w.proj_dtype, want_x_last=True)
    ref = oracle_forward_varying if w.varying_dt else oracle_forward
    oy, oxl = ref(inp)
    tol = BF16_TOL if (w.u_dtype == "bf16" or w.proj_dtype == "bf16") else FP32_TOL
    check(host(y), oy, tol, "y (%s, all sequences)" % name)
    check(host(xl), oxl, tol, "x_last (%s)" % name)
