"""Pins of the oracle's discretisation options, streaming step and
bidirectional layer, and of the HiPPO-N initialiser.

None of these checks calls the CUDA path.  Each compares with something
computed another way: the values the S4 page prints for the bilinear map, the
HiPPO-N eigenvalues it prints at N = 8, closed forms, a scipy ODE integrator,
explicit sums written out in numpy, and the (separately pinned) time-invariant
forward.
"""
import numpy as np
import pytest

import oracle
from _golden import read_golden
from diagonal_state_space_gb300 import init as s5init

scipy_integrate = pytest.importorskip("scipy.integrate")


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# Bilinear transform (S4 page, "Discretization and the step size Δ": two real
# eigenvalues at Delta = 0.1 and the values the page gives for their images,
# kept with the citation in tests/golden/s4_bilinear_examples.txt).
# --------------------------------------------------------------------------
def test_bilinear_matches_the_values_printed_on_the_s4_page():
    g = read_golden("s4_bilinear_examples.txt")
    lam = np.array([float(v) for v in g["lambda"]], dtype=np.complex128)
    step = float(g["step"][0])
    lb, bb = oracle.discretize_ex(lam, np.log(np.full(lam.size, step)), np.ones((lam.size, 1)),
                                  method="bilinear")
    for got, printed, nd in zip(lb, g["lambda_bar_bilinear"], g["printed_decimals"]):
        assert round(got.real, int(nd)) == float(printed) and abs(got.imag) == 0.0
    # the stable region: every Re(lambda) < 0 maps into the open unit disk (the page's claim)
    rng = _rng(1)
    lam = -rng.uniform(1e-3, 100, 200) + 1j * rng.uniform(-100, 100, 200)
    lb, _ = oracle.discretize_ex(lam, np.log(rng.uniform(1e-3, 10, 200)), np.ones((200, 1)), method="bilinear")
    assert np.all(np.abs(lb) < 1.0)


def test_bilinear_agrees_with_zoh_to_third_order_and_with_its_closed_form():
    rng = _rng(2)
    P, H = 40, 3
    lam = -rng.uniform(0.1, 1.0, P) + 1j * rng.uniform(-3, 3, P)
    dt = np.full(P, 1e-2)
    bt = rng.standard_normal((P, H)) + 1j * rng.standard_normal((P, H))
    lb_b, bb_b = oracle.discretize_ex(lam, np.log(dt), bt, method="bilinear")
    lb_z, bb_z = oracle.discretize_ex(lam, np.log(dt), bt, method="zoh")
    z = lam * dt
    # (1 + z/2)/(1 - z/2) - e^z = z^3/12 + O(z^4)
    assert np.allclose(lb_b - lb_z, z ** 3 / 12, rtol=0.05, atol=1e-12)
    # gain written out: dt / (1 - z/2)
    assert np.allclose(bb_b, (dt / (1 - z / 2))[:, None] * bt, rtol=1e-14, atol=0)
    # gain at lambda = 0 tends to dt, as the zero-order hold's does
    lb0, bb0 = oracle.discretize_ex(np.array([0j]), np.log([0.3]), np.ones((1, 1)), method="bilinear")
    assert lb0[0] == 1.0 and abs(bb0[0, 0] - 0.3) < 1e-15


def test_bilinear_recurrence_is_the_trapezoidal_rule_on_the_ode():
    # x' = lambda x + b u with u held piecewise linear between samples: the
    # trapezoidal rule integrates it exactly for a constant input.  Compare a
    # long constant-input run with the ODE solution at the same times.
    lam, dt, b = -0.7 + 2.0j, 0.01, 1.3 - 0.4j
    lb, bb = oracle.discretize_ex(np.array([lam]), np.log([dt]), np.array([[b]]), method="bilinear")
    # constant input u = 1 for 400 steps, zero state
    x = 0j
    for _ in range(400):
        x = lb[0] * x + bb[0, 0] * 1.0
    # trapezoid steady state equals the continuous one, -b/lambda; the transient
    # decays as lambda_bar^k, so compare with the exact continuous solution
    t = 400 * dt
    exact = -b / lam * (1 - np.exp(lam * t))
    assert abs(x - exact) < 5e-4 * abs(exact)


# --------------------------------------------------------------------------
# clip_eigs and sampling-rate rescaling.
# --------------------------------------------------------------------------
def test_clip_eigs_clips_only_real_parts_above_the_threshold():
    lam = np.array([0.3 + 2j, -1e-5 - 1j, -0.5 + 0.5j])
    dt = np.array([0.05, 0.05, 0.05])
    lb, _ = oracle.discretize_ex(lam, np.log(dt), np.ones((3, 1)), clip_re=-1e-4)
    expect = np.exp(np.array([-1e-4 + 2j, -1e-4 - 1j, -0.5 + 0.5j]) * dt)
    assert np.allclose(lb, expect, rtol=1e-15, atol=0)


def test_rate_rescaling_doubles_the_interval_from_16_to_8_khz():
    # review "Sampling intervals carry physical meaning": old rate / new rate
    lam = np.array([-1.0 + 0j, -0.5 + 3j])
    lb, bb = oracle.discretize_ex(lam, np.log([0.1, 0.02]), np.ones((2, 1)), dt_scale=16000 / 8000)
    assert np.allclose(lb, np.exp(lam * np.array([0.2, 0.04])), rtol=1e-15, atol=0)
    assert np.allclose(bb[:, 0], (np.exp(lam * np.array([0.2, 0.04])) - 1) / lam, rtol=1e-14, atol=0)


def test_zoh_with_options_matches_ode_integration():
    lam, dt = -0.3 + 1.7j, 0.37
    lb, bb = oracle.discretize_ex(np.array([lam]), np.log([dt / 3]), np.array([[1.0 + 0j]]), dt_scale=3.0)
    sol = scipy_integrate.solve_ivp(lambda t, v: [lam * v[0] + 1.0], (0, dt), [0j], rtol=1e-12, atol=1e-14)
    assert abs(sol.y[0, -1] - bb[0, 0]) < 1e-9
    sol = scipy_integrate.solve_ivp(lambda t, v: [lam * v[0]], (0, dt), [1 + 0j], rtol=1e-12, atol=1e-14)
    assert abs(sol.y[0, -1] - lb[0]) < 1e-9


# --------------------------------------------------------------------------
# Streaming step: L steps equal the (pinned) forward over L tokens.
# --------------------------------------------------------------------------
def test_steps_equal_the_forward_pass():
    rng = _rng(3)
    B, L, H, P = 3, 17, 5, 4
    lb = rng.uniform(0.3, 0.99, P) * np.exp(1j * rng.uniform(-3, 3, P))
    bb = rng.standard_normal((P, H)) + 1j * rng.standard_normal((P, H))
    ct = rng.standard_normal((H, P)) + 1j * rng.standard_normal((H, P))
    d = rng.standard_normal(H)
    u = rng.standard_normal((B, L, H))
    x0 = rng.standard_normal((B, P)) + 1j * rng.standard_normal((B, P))
    y_ref, xl = oracle.forward(lb, bb, ct, d, u, x0=x0)
    x = x0.copy()
    for k in range(L):
        x, yk = oracle.step(lb, bb, ct, d, x, u[:, k])
        assert np.allclose(yk, y_ref[:, k], rtol=1e-12, atol=1e-12)
    assert np.allclose(x, xl, rtol=1e-12, atol=1e-12)
    # one step written out
    x1, y1 = oracle.step(lb, bb, ct, d, x0, u[:, 0])
    xe = lb * x0 + u[:, 0] @ bb.T
    assert np.allclose(x1, xe, rtol=1e-13, atol=1e-13)
    assert np.allclose(y1, 2 * np.real(xe @ ct.T) + d * u[:, 0], rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# Bidirectional layer: explicit sums over past and future inputs.
# --------------------------------------------------------------------------
def test_bidirectional_equals_explicit_sums():
    rng = _rng(4)
    B, L, H, P = 2, 9, 4, 3
    lb = rng.uniform(0.3, 0.95, P) * np.exp(1j * rng.uniform(-3, 3, P))
    bb = rng.standard_normal((P, H)) + 1j * rng.standard_normal((P, H))
    c2 = rng.standard_normal((H, 2 * P)) + 1j * rng.standard_normal((H, 2 * P))
    d = rng.standard_normal(H)
    u = rng.standard_normal((B, L, H))
    y = oracle.forward_bidirectional(lb, bb, c2, d, u)
    bu = np.einsum("ph,blh->blp", bb, u)
    ye = np.empty_like(y)
    for b in range(B):
        for k in range(L):
            xf = sum(lb ** (k - j) * bu[b, j] for j in range(0, k + 1))
            xb = sum(lb ** (j - k) * bu[b, j] for j in range(k, L))
            ye[b, k] = 2 * np.real(c2[:, :P] @ xf + c2[:, P:] @ xb) + d * u[b, k]
    assert np.allclose(y, ye, rtol=1e-12, atol=1e-12)
    # with the backward half of C~ zero it is the causal layer
    c2f = c2.copy()
    c2f[:, P:] = 0
    assert np.allclose(oracle.forward_bidirectional(lb, bb, c2f, d, u),
                       oracle.forward(lb, bb, c2[:, :P], d, u)[0], rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# HiPPO-N (review row 5; summary App. B.1.1; S4 page "Normal plus low-rank").
# --------------------------------------------------------------------------
def test_hippo_normal_structure_and_the_eigenvalues_printed_at_n8():
    a = s5init.hippo_normal(8)
    assert np.all(np.diag(a) == -0.5)
    off = a + 0.5 * np.eye(8)
    assert np.allclose(off, -off.T, atol=0)
    assert a[0, 1] == np.sqrt(0.5 * 1.5) and a[1, 0] == -np.sqrt(0.5 * 1.5)
    # HiPPO-LegS (-(n+1) on the diagonal, -sqrt(2n+1)sqrt(2k+1) below, 0 above)
    # plus (1/2) P P^T with P_n = sqrt(2n+1) is exactly HiPPO-N
    n = np.arange(8)
    legs = -np.tril(np.sqrt(np.outer(2 * n + 1, 2 * n + 1)), -1) - np.diag(n + 1.0)
    pp = 0.5 * np.outer(np.sqrt(2 * n + 1), np.sqrt(2 * n + 1))
    assert np.allclose(legs + pp, a, rtol=0, atol=1e-14)
    g = read_golden("hippo_n_n8_eigenvalues.txt")
    assert int(g["n"][0]) == 8
    ev, v = s5init.hippo_normal_eig(8)
    assert np.allclose(ev.real, float(g["real_part"][0]), atol=1e-12)
    printed = np.array([float(x) for x in g["imag_abs_descending"]])
    got = np.sort(np.abs(ev.imag))[::-1][::2]
    assert np.allclose(np.round(got, int(g["decimals"][0])), printed, atol=0)
    assert np.allclose(v @ np.diag(ev) @ v.conj().T, a, atol=1e-12)
    assert np.allclose(np.linalg.eigvals(a).real, -0.5, atol=1e-9)


def test_hippo_init_half_spectrum_reproduces_the_full_real_system():
    P, H = 6, 5
    lam, log_dt, bt, ct, d = s5init.init_s5(P, H, seed=3)
    assert lam.shape == (P,) and bt.shape == (P, H) and ct.shape == (H, P)
    assert np.all(lam.imag >= 0) and np.allclose(lam.real, -0.5, atol=1e-6)
    # continuous impulse responses: full real system C e^{At} B versus the
    # stored half spectrum 2 Re(C~ e^{Lambda t} B~)
    rng = np.random.default_rng(3)
    n = 2 * P
    b_full = rng.standard_normal((n, H)) / np.sqrt(H)
    c_full = rng.standard_normal((H, n)) / np.sqrt(n)
    a = s5init.hippo_normal(n)
    for t in (0.0, 0.3, 1.7):
        w, vec = np.linalg.eig(a * t)
        eat = (vec @ np.diag(np.exp(w)) @ np.linalg.inv(vec)).real
        full = c_full @ eat @ b_full
        half = 2 * np.real(ct.astype(np.complex128) @ np.diag(np.exp(lam.astype(np.complex128) * t)) @ bt.astype(np.complex128))
        assert np.allclose(full, half, rtol=1e-4, atol=1e-5)
