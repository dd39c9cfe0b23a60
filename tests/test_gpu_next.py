"""GPU parity of the options and variants beyond the causal layer: the
discretisation options (bilinear, clip_eigs, rate rescaling), the streaming
step, the bidirectional layer, and a forward pass from the HiPPO-N
initialiser.  CUDA path through the C ABI against the float64 oracle on the
same seeded inputs.

Bars: discretisation is float64 on the device rounded once (2e-7 relative per
element); float32 paths 1e-5 relative L2 per output tensor; bf16 paths 2e-2.
"""
import numpy as np
import pytest
import torch

from diagonal_state_space_gb300 import api
from diagonal_state_space_gb300 import init as s5init
from diagonal_state_space_gb300._native import S5Error
from diagonal_state_space_gb300.workloads import WORKLOADS, bf16_round, make_inputs, make_layer_inputs

from _parity import check, dev, host, layer_to_device
import oracle

pytestmark = pytest.mark.gpu

FP32_TOL = 1e-5
BF16_TOL = 2e-2


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    torch.cuda.init()


# --------------------------------------------------------------------------
# discretisation options
# --------------------------------------------------------------------------
@pytest.mark.parametrize("method", ["zoh", "bilinear"])
@pytest.mark.parametrize("clip_re,dt_scale", [(0.0, 1.0), (-1e-4, 1.0), (0.0, 2.0), (-1e-4, 0.5)])
@pytest.mark.parametrize("P,H", [(1, 1), (64, 128), (300, 7)])
def test_discretize_ex_matches_oracle(method, clip_re, dt_scale, P, H):
    inp = make_layer_inputs(1, 1, H, P, seed=11 + P + H)
    lam = inp["lambda_"].copy()
    lam[::3] = (np.abs(lam[::3].real) * 0.5 + 1j * lam[::3].imag).astype(np.complex64)  # some Re > 0: clipped
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize_ex(dev(lam), t["log_dt"], t["b_tilde"], method, clip_re, dt_scale)
    olb, obb = oracle.discretize_ex(lam, inp["log_dt"], inp["b_tilde"], method, clip_re,
                                    float(np.float32(dt_scale)))
    np.testing.assert_allclose(host(lb), olb, rtol=2e-7, atol=1e-30)
    np.testing.assert_allclose(host(bb), obb, rtol=3e-7, atol=1e-12 * np.max(np.abs(obb)))


def test_discretize_ex_zoh_equals_discretize():
    inp = make_layer_inputs(1, 1, 48, 40, seed=3)
    t = layer_to_device(inp)
    a = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    b = api.s5_discretize_ex(t["lam"], t["log_dt"], t["b_tilde"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_discretize_ex_rejects_bad_options():
    inp = make_layer_inputs(1, 1, 8, 4, seed=3)
    t = layer_to_device(inp)
    for kw in (dict(dt_scale=0.0), dict(dt_scale=-1.0), dict(clip_re=1e-3)):
        with pytest.raises(S5Error):
            api.s5_discretize_ex(t["lam"], t["log_dt"], t["b_tilde"], **kw)


# --------------------------------------------------------------------------
# streaming step
# --------------------------------------------------------------------------
# several sequence groups (B > 8, ragged), P and H not multiples of 8, and a
# size whose staged states need more than 48 KiB of shared memory
@pytest.mark.parametrize("B,H,P,steps", [(1, 1, 1, 3), (3, 32, 16, 20), (8, 128, 128, 8), (2, 300, 70, 5),
                                         (19, 64, 40, 3), (2, 1024, 1024, 2)])
def test_step_matches_oracle(B, H, P, steps):
    inp = make_layer_inputs(B, steps, H, P, seed=21 + H)
    olb, obb = oracle.discretize(inp["lambda_"], inp["log_dt"], inp["b_tilde"])
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    rng = np.random.default_rng(5)
    x0 = (rng.standard_normal((B, P)) + 1j * rng.standard_normal((B, P))).astype(np.complex64)
    x = dev(x0)
    ox = x0.astype(np.complex128)
    for k in range(steps):
        uk = np.ascontiguousarray(inp["u"][:, k])
        y = api.s5_step(lb, bb, t["c_tilde"], t["d"], x, dev(uk))
        ox, oy = oracle.step(olb, obb, inp["c_tilde"], inp["d"], ox, uk)
        check(host(y), oy, FP32_TOL, "host(y)")
        # the D*u-free part alone
        check(host(y) - inp["d"] * uk, oy - inp["d"] * uk, FP32_TOL, "host(y) - inp['d'] * uk")
    check(host(x), ox, FP32_TOL, "host(x)")


def test_steps_continue_a_forward_pass():
    B, L, H, P = 2, 37, 32, 16
    inp = make_layer_inputs(B, L + 4, H, P, seed=9)
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    y_all = api.s5_forward(lb, bb, t["c_tilde"], t["d"], t["u"])
    _, xl = api.s5_forward(lb, bb, t["c_tilde"], t["d"], t["u"][:, :L].contiguous(), x_last=True)
    for k in range(L, L + 4):
        yk = api.s5_step(lb, bb, t["c_tilde"], t["d"], xl, t["u"][:, k].contiguous())
        check(host(yk), host(y_all[:, k]), FP32_TOL, "host(yk)")


def test_back_to_back_steps_match_synchronised_steps():
    """Streaming steps launched back to back (each may be scheduled while the
    one before finishes, and reads the state that one writes) give, bit for
    bit, what the same steps give with the device synchronised after each."""
    B, H, P, n = 8, 128, 128, 24
    inp = make_layer_inputs(B, n, H, P, seed=77)
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    u = [t["u"][:, k].contiguous() for k in range(n)]
    torch.cuda.synchronize()

    def steps(sync):
        x = torch.zeros(B, P, dtype=torch.complex64, device="cuda")
        ys = []
        for k in range(n):
            ys.append(api.s5_step(lb, bb, t["c_tilde"], t["d"], x, u[k]))
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return [host(y) for y in ys], host(x)

    chained, xc = steps(sync=False)
    synced, xs = steps(sync=True)
    assert np.array_equal(xc, xs)
    for a, b in zip(chained, synced):
        assert np.array_equal(a, b)


def test_step_rejects_misaligned_and_empty_batch_is_a_noop():
    inp = make_layer_inputs(2, 1, 8, 4, seed=3)
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    x = torch.zeros(2, 4, dtype=torch.complex64, device="cuda")
    u = torch.zeros(2 * 8 + 1, dtype=torch.float32, device="cuda")[1:].view(2, 8)
    with pytest.raises(S5Error):
        api.s5_step(lb, bb, t["c_tilde"], t["d"], x, u)
    x0 = torch.zeros(0, 4, dtype=torch.complex64, device="cuda")
    y0 = api.s5_step(lb, bb, t["c_tilde"], t["d"], x0, torch.zeros(0, 8, device="cuda"))
    assert y0.shape == (0, 8)


# --------------------------------------------------------------------------
# bidirectional layer
# --------------------------------------------------------------------------
def _c2(inp, seed):
    rng = np.random.default_rng(seed)
    H, P = inp["c_tilde"].shape
    cb = ((rng.standard_normal((H, P)) + 1j * rng.standard_normal((H, P))) / np.sqrt(2 * H)).astype(np.complex64)
    return np.ascontiguousarray(np.concatenate([inp["c_tilde"], cb], axis=1))


@pytest.mark.parametrize("B,L,H,P", [(1, 1, 8, 4), (2, 77, 32, 16), (3, 300, 64, 24), (1, 1000, 128, 64)])
def test_bidirectional_f32_matches_oracle(B, L, H, P):
    inp = make_layer_inputs(B, L, H, P, seed=31 + L)
    c2 = _c2(inp, L)
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    olb, obb = oracle.discretize(inp["lambda_"], inp["log_dt"], inp["b_tilde"])
    for dz in (False, True):
        d = np.zeros_like(inp["d"]) if dz else inp["d"]
        y = api.s5_forward_bidirectional(lb, bb, dev(c2), dev(d), t["u"])
        oy = oracle.forward_bidirectional(olb, obb, c2, d, inp["u"])
        check(host(y), oy, FP32_TOL, "host(y)")


# ragged last chunk (the backward scan's first), many lanes per sequence, one
# lane per sequence (B = 60), several sequences per CTA (B = 160)
@pytest.mark.parametrize("B,L", [(2, 700), (1, 4096), (1, 1), (60, 130), (160, 65)])
def test_bidirectional_bf16_tensor_core_path_matches_oracle(B, L):
    H = P = 128
    inp = make_layer_inputs(B, L, H, P, seed=41 + L, u_dtype="bf16")
    c2 = _c2(inp, L)
    t = layer_to_device(inp, "bf16")
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    y = api.s5_forward_bidirectional(lb, bb, dev(c2), t["d"], t["u"], proj_dtype="bf16")
    assert y.dtype == torch.bfloat16
    olb, obb = oracle.discretize(inp["lambda_"], inp["log_dt"], inp["b_tilde"])
    oy = oracle.forward_bidirectional(olb, obb, c2, inp["d"], inp["u"])
    check(host(y.float()), oy, BF16_TOL, "host(y.float())")
    # the SSM terms alone (D = 0)
    y0 = api.s5_forward_bidirectional(lb, bb, dev(c2), dev(np.zeros(H, np.float32)), t["u"], proj_dtype="bf16")
    oy0 = oracle.forward_bidirectional(olb, obb, c2, np.zeros(H), inp["u"])
    check(host(y0.float()), oy0, BF16_TOL, "host(y0.float())")


def test_bidirectional_with_zero_backward_half_is_the_causal_layer():
    B, L, H, P = 2, 200, 32, 16
    inp = make_layer_inputs(B, L, H, P, seed=5)
    c2 = np.ascontiguousarray(np.concatenate([inp["c_tilde"], np.zeros_like(inp["c_tilde"])], axis=1))
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    yb = api.s5_forward_bidirectional(lb, bb, dev(c2), t["d"], t["u"])
    yf = api.s5_forward(lb, bb, t["c_tilde"], t["d"], t["u"])
    check(host(yb), host(yf), 1e-6, "host(yb)")


# --------------------------------------------------------------------------
# HiPPO-N initialisation through the layer
# --------------------------------------------------------------------------
def test_forward_from_hippo_init_matches_oracle():
    B, L, H, P = 2, 300, 32, 16
    lam, log_dt, bt, ct, d = s5init.init_s5(P, H, blocks=2, seed=7)
    rng = np.random.default_rng(7)
    u = rng.standard_normal((B, L, H)).astype(np.float32)
    lb, bb = api.s5_discretize(dev(lam), dev(log_dt), dev(bt))
    y = api.s5_forward(lb, bb, dev(ct), dev(d), dev(u))
    olb, obb = oracle.discretize(lam, log_dt, bt)
    oy, _ = oracle.forward(olb, obb, ct, d, u)
    check(host(y), oy, FP32_TOL, "host(y)")


# --------------------------------------------------------------------------
# The three NEXT-row benchmark workloads at full size, through the calls the
# benchmark times; the oracle computes every sequence.
# --------------------------------------------------------------------------
def test_full_size_bidirectional_workload():
    w = WORKLOADS["pathx_bf16_bidir"]
    inp = make_inputs(w)
    t = layer_to_device(inp, w.u_dtype)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    y = api.s5_forward_bidirectional(lb, bb, dev(inp["c_tilde2"]), t["d"], t["u"], proj_dtype="bf16")
    olb, obb = oracle.discretize(inp["lambda_"], inp["log_dt"], inp["b_tilde"])
    oy = oracle.forward_bidirectional(olb, obb, inp["c_tilde2"], inp["d"], inp["u"])
    check(host(y.float()), oy, BF16_TOL, "y (bidirectional, all sequences)")
    # the SSM terms alone
    du = inp["d"] * inp["u"].astype(np.float64)
    check(host(y.float()) - du, oy - du, BF16_TOL, "y - D u (bidirectional)")


def test_full_size_bilinear_workload():
    w = WORKLOADS["pathx_bf16_bilinear"]
    inp = make_inputs(w)
    t = layer_to_device(inp, w.u_dtype)
    lb, bb = api.s5_discretize_ex(t["lam"], t["log_dt"], t["b_tilde"], method=w.method, clip_re=w.clip_re,
                                  dt_scale=w.dt_scale)
    y, xl = api.s5_forward(lb, bb, t["c_tilde"], t["d"], t["u"], proj_dtype="bf16", x_last=True)
    olb, obb = oracle.discretize_ex(inp["lambda_"], inp["log_dt"], inp["b_tilde"], w.method,
                                    float(np.float32(w.clip_re)), float(np.float32(w.dt_scale)))
    oy, oxl = oracle.forward(olb, obb, inp["c_tilde"], inp["d"], inp["u"])
    check(host(y.float()), oy, BF16_TOL, "y (bilinear, all sequences)")
    check(host(xl), oxl, BF16_TOL, "x_last (bilinear)")


def test_full_size_streaming_workload():
    w = WORKLOADS["stream"]
    inp = make_inputs(w)
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    x = torch.zeros(w.B, w.P, dtype=torch.complex64, device="cuda")
    u_t = t["u"].transpose(0, 1).contiguous()          # [L, B, H]: one contiguous slice per call
    ys = [api.s5_step(lb, bb, t["c_tilde"], t["d"], x, u_t[k]) for k in range(w.L)]
    y = torch.stack(ys, dim=1)
    olb, obb = oracle.discretize(inp["lambda_"], inp["log_dt"], inp["b_tilde"])
    oy, oxl = oracle.forward(olb, obb, inp["c_tilde"], inp["d"], inp["u"])
    check(host(y), oy, FP32_TOL, "host(y)")
    check(host(y) - inp["d"] * inp["u"], oy - inp["d"] * inp["u"], FP32_TOL, "host(y) - inp['d'] * inp['u']")
    check(host(x), oxl, FP32_TOL, "host(x)")
