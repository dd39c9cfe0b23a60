"""Pins of the float64 oracle against what the pages and mathematics fix.

None of these checks calls the CUDA path.  Each one compares the oracle with
something computed another way: a brute-force associative scan, a library
linear filter (scipy.signal.lfilter), an ODE integrator (scipy solve_ivp),
closed forms, the worked example printed on the S4 page, finite differences,
and PyTorch's own LayerNorm / GELU / sigmoid routines.
"""
from fractions import Fraction
from functools import lru_cache

import numpy as np
import pytest

import oracle
from _golden import read_golden

scipy_signal = pytest.importorskip("scipy.signal")
scipy_integrate = pytest.importorskip("scipy.integrate")



def _rng(seed):
    return np.random.default_rng(seed)


def _rand_system(rng, H, P, stable=True):
    """Random discrete diagonal system (lambda_bar inside the unit disk)."""
    r = rng.uniform(0.3, 0.99, P) if stable else rng.uniform(0.5, 1.5, P)
    th = rng.uniform(-np.pi, np.pi, P)
    lb = r * np.exp(1j * th)
    bb = rng.standard_normal((P, H)) + 1j * rng.standard_normal((P, H))
    ct = rng.standard_normal((H, P)) + 1j * rng.standard_normal((H, P))
    d = rng.standard_normal(H)
    return lb, bb, ct, d


# --------------------------------------------------------------------------
# Scan: the sequential recurrence equals every associative bracketing.
# ("S5: Simplified State Space Layers..." review, "Associative scans preserve
# the recurrence" and row 3; summary App. H.)
# --------------------------------------------------------------------------
def _compose(e, l):
    """Earlier element e = (a_i, b_i), later l = (a_j, b_j): x -> a_j (a_i x + b_i) + b_j."""
    return (l[0] * e[0], l[0] * e[1] + l[1])


def _recursive_prefix(items):
    """Pair neighbours, scan the pairs recursively, then fill in the odd positions."""
    if len(items) <= 1:
        return list(items)
    pairs = [_compose(items[i], items[i + 1]) for i in range(0, len(items) - 1, 2)]
    pre = _recursive_prefix(pairs)
    out = []
    for i, it in enumerate(items):
        if i == 0:
            out.append(it)
        elif i % 2 == 1:
            out.append(pre[i // 2])
        else:
            out.append(_compose(pre[i // 2 - 1], it))
    return out


@lru_cache(maxsize=None)
def _bracketings(i, j):
    """All binary trees over the contiguous range [i, j)."""
    if j - i == 1:
        return [i]
    trees = []
    for m in range(i + 1, j):
        for left in _bracketings(i, m):
            for right in _bracketings(m, j):
                trees.append((left, right))
    return trees


def _eval_tree(tree, items):
    if isinstance(tree, int):
        return items[tree]
    return _compose(_eval_tree(tree[0], items), _eval_tree(tree[1], items))


@pytest.mark.parametrize("L", [1, 2, 3, 5, 6, 7, 8, 13])
def test_recurrence_equals_associative_scan(L):
    rng = _rng(L)
    H, P = 3, 4
    lb, bb, ct, d = _rand_system(rng, H, P)
    u = rng.standard_normal((1, L, H))
    _, states = oracle.forward(lb, bb, ct, d, u, return_states=True)
    bu = u[0] @ bb.T                                        # b_k = B_bar u_k
    items = [(lb.copy(), bu[k]) for k in range(L)]
    pre = _recursive_prefix(items)
    for k in range(L):
        np.testing.assert_allclose(states[0, k], pre[k][1], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(pre[k][0], lb ** (k + 1), rtol=1e-13)
    if L <= 6:
        for tree in _bracketings(0, L):
            a, b = _eval_tree(tree, items)
            np.testing.assert_allclose(b, states[0, L - 1], rtol=1e-13, atol=1e-13)


def _lfilter_full_spectrum(lb, bb, ct, d, u):
    """Library recurrence (scipy lfilter) on the full conjugate-pair system; the
    real output is the plain sum over both members of every pair."""
    Bn, L, H = u.shape
    y = np.empty((Bn, L, H))
    for b in range(Bn):
        bu = u[b] @ bb.T
        x = np.stack([scipy_signal.lfilter([1.0], [1.0, -lb[p]], bu[:, p])
                      for p in range(len(lb))], axis=1)      # [L, P]
        full = x @ ct.T + np.conj(x) @ np.conj(ct).T          # both pair members
        assert np.max(np.abs(full.imag)) < 1e-9 * max(1.0, np.max(np.abs(full.real)))
        y[b] = full.real + d * u[b]
    return y


@pytest.mark.parametrize("B,L,H,P", [(1, 1, 1, 1), (2, 37, 5, 3), (3, 64, 8, 6)])
def test_half_spectrum_readout_equals_full_conjugate_system(B, L, H, P):
    """Review row 4 and wiki 'Paper vs code': with only one member of each
    conjugate pair stored, 2*Re(C x) equals the full system's real output."""
    rng = _rng(100 + L)
    lb, bb, ct, d = _rand_system(rng, H, P)
    u = rng.standard_normal((B, L, H))
    y, _ = oracle.forward(lb, bb, ct, d, u)
    np.testing.assert_allclose(y, _lfilter_full_spectrum(lb, bb, ct, d, u), rtol=1e-11, atol=1e-11)


def test_constant_input_geometric_series():
    """Constant input: x_k = b (1 - a^k) / (1 - a) (geometric series)."""
    rng = _rng(7)
    H, P, L = 4, 5, 50
    lb, bb, ct, d = _rand_system(rng, H, P)
    u1 = rng.standard_normal(H)
    u = np.broadcast_to(u1, (1, L, H)).copy()
    _, st = oracle.forward(lb, bb, ct, d, u, return_states=True)
    b = bb @ u1
    k = np.arange(1, L + 1)[:, None]
    closed = b * (1 - lb ** k) / (1 - lb)
    np.testing.assert_allclose(st[0], closed, rtol=1e-12, atol=1e-12)


def test_impulse_response_is_convolution_kernel():
    """Convolution view (S4 page, 'How a state space model works'; textbook
    section 13.1): an impulse at step 1 gives y_k = 2 Re(C lb^(k-1) B e_h) + D_h [k=1]."""
    rng = _rng(8)
    H, P, L = 3, 4, 20
    lb, bb, ct, d = _rand_system(rng, H, P)
    for h in range(H):
        u = np.zeros((1, L, H))
        u[0, 0, h] = 1.0
        y, _ = oracle.forward(lb, bb, ct, d, u)
        kern = np.stack([(ct * (lb ** i)) @ bb[:, h] for i in range(L)])   # [L, H] complex
        expect = 2 * kern.real
        expect[0, h] += d[h]
        np.testing.assert_allclose(y[0], expect, rtol=1e-12, atol=1e-12)




def test_s4_page_worked_example_scalar_pulse():
    """The S4 page's hand-computed example: x_k = x_{k-1}/3 + 2u_k/3, kernel
    (2/3)(1/3)^i, pulse (1,1,1,1,0,0,0,0).  Reached through the zero-order hold
    with a real pole lambda = -ln 3, interval 1 and B~ = ln 3 (so lambda_bar = 1/3
    and B_bar = 2/3), and C~ = 1/2 so that the factor-2 readout reads x itself."""
    g = read_golden("s4_scalar_pulse.txt")
    pulse = [int(v) for v in g["pulse"]]
    kern = [Fraction(int(n), int(dn)) for n, dn in zip(g["kernel_num"], g["kernel_den"])]
    L = len(pulse)
    expect = [sum(kern[k - j] * pulse[j] for j in range(k + 1)) for k in range(L)]
    lam = np.array([-np.log(3.0) + 0j])
    lb, bb = oracle.discretize(lam, np.array([0.0]), np.array([[np.log(3.0) + 0j]]))
    assert abs(lb[0] - Fraction(g["recurrence_a"][0])) < 1e-15
    assert abs(bb[0, 0] - float(Fraction(g["recurrence_b"][0]))) < 1e-15
    u = np.array(pulse, dtype=np.float64).reshape(1, L, 1)
    y, _ = oracle.forward(lb, bb, np.array([[0.5 + 0j]]), np.array([0.0]), u)
    np.testing.assert_allclose(y[0, :, 0], [float(e) for e in expect], rtol=1e-14, atol=1e-15)
    # first values by hand: 2/3, 8/9, 26/27, 80/81, then a factor 1/3 per step
    assert expect[:5] == [Fraction(2, 3), Fraction(8, 9), Fraction(26, 27), Fraction(80, 81),
                          Fraction(80, 243)]


# --------------------------------------------------------------------------
# Zero-order hold: exact integration of a held input (review
# "Discretization controls both retention and input gain", row 2; summary
# section 3.2 eq. 6).
# --------------------------------------------------------------------------
def _ode_step(lam, bt_u, x0, dt):
    """Integrate dx/dt = lam x + bt_u from x0 over [0, dt] (real 2-vector form)."""
    def f(_t, v):
        x = v[0] + 1j * v[1]
        dx = lam * x + bt_u
        return [dx.real, dx.imag]
    if dt == 0:
        return x0
    sol = scipy_integrate.solve_ivp(f, (0.0, dt), [x0.real, x0.imag], method="DOP853",
                                    rtol=1e-12, atol=1e-14)
    return sol.y[0, -1] + 1j * sol.y[1, -1]


def test_zoh_matches_ode_integration():
    rng = _rng(11)
    P, H = 6, 3
    lam = -rng.uniform(0.05, 2.0, P) + 1j * rng.uniform(-30, 30, P)
    log_dt = rng.uniform(np.log(1e-3), np.log(0.5), P)
    bt = rng.standard_normal((P, H)) + 1j * rng.standard_normal((P, H))
    lb, bb = oracle.discretize(lam, log_dt, bt)
    u = rng.standard_normal(H)
    x0 = rng.standard_normal(P) + 1j * rng.standard_normal(P)
    for p in range(P):
        ref = _ode_step(lam[p], bt[p] @ u, x0[p], np.exp(log_dt[p]))
        got = lb[p] * x0[p] + bb[p] @ u
        assert abs(got - ref) <= 1e-9 * max(1.0, abs(ref))


def test_zoh_half_steps_compose_to_full_step():
    rng = _rng(12)
    P, H = 5, 4
    lam = -rng.uniform(0.1, 1.0, P) + 1j * rng.uniform(-10, 10, P)
    log_dt = rng.uniform(np.log(1e-3), np.log(0.1), P)
    bt = rng.standard_normal((P, H)) + 1j * rng.standard_normal((P, H))
    lb1, bb1 = oracle.discretize(lam, log_dt, bt)
    lbh, bbh = oracle.discretize(lam, log_dt - np.log(2.0), bt)
    np.testing.assert_allclose(lbh ** 2, lb1, rtol=1e-13)
    np.testing.assert_allclose(lbh[:, None] * bbh + bbh, bb1, rtol=1e-11, atol=1e-14)


def test_zero_pole_and_small_interval_limits():
    """Review row 2: the input gain tends to dt at a zero pole (phi1(0) = 1)."""
    bt = np.array([[1.0 + 2.0j, -0.5 + 0.25j]])
    lb, bb = oracle.discretize(np.array([0.0 + 0.0j]), np.array([np.log(0.37)]), bt)
    assert lb[0] == 1.0
    np.testing.assert_allclose(bb, 0.37 * bt, rtol=1e-15)
    lam = np.array([-0.5 + 3.0j])
    for dt in (1e-6, 1e-9, 1e-12):
        lb, bb = oracle.discretize(lam, np.array([np.log(dt)]), bt)
        np.testing.assert_allclose(bb / (dt * bt), 1.0, rtol=2 * abs(lam[0]) * dt + 1e-13)
        np.testing.assert_allclose(lb[0], 1.0, atol=2 * abs(lam[0]) * dt)
    # series and quotient branches agree at the switch point |z| = 1e-4
    for zabs in (0.999999e-4, 1.000001e-4):
        dt = zabs / abs(lam[0])
        lb, bb = oracle.discretize(lam, np.array([np.log(dt)]), bt)
        exact = np.expm1(lam[0] * dt) / lam[0]       # complex expm1 via numpy
        np.testing.assert_allclose(bb[0] / bt[0], exact, rtol=1e-11)


# --------------------------------------------------------------------------
# Irregular sampling (summary section 3.3 / 6.3; review "Sampling intervals
# carry physical meaning").
# --------------------------------------------------------------------------
def _state_readout(P):
    """C~ [2P, P] with 2 Re(C~ x): rows 2p -> Re x_p, rows 2p+1 -> Im x_p."""
    ct = np.zeros((2 * P, P), complex)
    for p in range(P):
        ct[2 * p, p] = 0.5
        ct[2 * p + 1, p] = -0.5j
    return ct


def test_varying_dt_matches_ode_over_irregular_intervals():
    rng = _rng(21)
    P, L = 3, 7
    H = 2 * P
    lam = -rng.uniform(0.1, 1.0, P) + 1j * rng.uniform(-8, 8, P)
    log_dt = rng.uniform(np.log(0.01), np.log(0.3), P)
    bt = rng.standard_normal((P, H)) + 1j * rng.standard_normal((P, H))
    g = rng.exponential(1.0, (1, L))
    g[0, 3] = 0.0
    u = rng.standard_normal((1, L, H))
    x0 = rng.standard_normal((1, P)) + 1j * rng.standard_normal((1, P))
    y, xl = oracle.forward_varying_dt(lam, log_dt, bt, _state_readout(P), np.zeros(H), g, u, x0)
    x = x0[0].copy()
    for k in range(L):
        for p in range(P):
            x[p] = _ode_step(lam[p], bt[p] @ u[0, k], x[p], g[0, k] * np.exp(log_dt[p]))
        np.testing.assert_allclose(y[0, k, 0::2], x.real, rtol=1e-8, atol=1e-10)
        np.testing.assert_allclose(y[0, k, 1::2], x.imag, rtol=1e-8, atol=1e-10)
    np.testing.assert_allclose(xl[0], x, rtol=1e-8, atol=1e-10)


def test_zero_gap_leaves_state_unchanged():
    rng = _rng(22)
    P, L = 4, 9
    H = 2 * P
    lam = -0.5 + 1j * np.pi * np.arange(P)
    log_dt = rng.uniform(np.log(1e-3), np.log(1e-1), P)
    bt = rng.standard_normal((P, H)) + 1j * rng.standard_normal((P, H))
    u = rng.standard_normal((1, L, H))
    g = rng.exponential(1.0, (1, L))
    g[0, 4] = 0.0
    y, _ = oracle.forward_varying_dt(lam, log_dt, bt, _state_readout(P), np.zeros(H), g, u)
    np.testing.assert_array_equal(y[0, 4], y[0, 3])        # x_5 = x_4 exactly
    assert np.all(y[0, 5] != y[0, 4])
    x0 = rng.standard_normal((1, P)) + 1j * rng.standard_normal((1, P))
    _, xl = oracle.forward_varying_dt(lam, log_dt, bt, _state_readout(P), np.zeros(H),
                                      np.zeros((1, L)), u, x0)
    np.testing.assert_array_equal(xl, x0)


def test_unit_gaps_equal_time_invariant_layer():
    rng = _rng(23)
    P, H, L, B = 5, 6, 33, 2
    lam = -0.5 + 1j * np.pi * np.arange(P)
    log_dt = rng.uniform(np.log(1e-3), np.log(1e-1), P)
    bt = rng.standard_normal((P, H)) + 1j * rng.standard_normal((P, H))
    ct = rng.standard_normal((H, P)) + 1j * rng.standard_normal((H, P))
    d = rng.standard_normal(H)
    u = rng.standard_normal((B, L, H))
    yv, xv = oracle.forward_varying_dt(lam, log_dt, bt, ct, d, np.ones((B, L)), u)
    # ZOH by the ODE solution: lambda_bar = exp(lam dt), gain from solve_ivp
    dt = np.exp(log_dt)
    lb = np.exp(lam * dt)
    gain = np.array([_ode_step(lam[p], 1.0, 0.0, dt[p]) for p in range(P)])
    y_ref = _lfilter_full_spectrum(lb, gain[:, None] * bt, ct, d, u)
    np.testing.assert_allclose(yv, y_ref, rtol=1e-8, atol=1e-9)


def test_streaming_in_two_calls_equals_one_call():
    """Review 'Associative scans': a non-zero initial state continues the sequence."""
    rng = _rng(31)
    lb, bb, ct, d = _rand_system(rng, 4, 3)
    u = rng.standard_normal((2, 40, 4))
    y, xl = oracle.forward(lb, bb, ct, d, u)
    y1, x1 = oracle.forward(lb, bb, ct, d, u[:, :17])
    y2, x2 = oracle.forward(lb, bb, ct, d, u[:, 17:], x0=x1)
    np.testing.assert_allclose(np.concatenate([y1, y2], 1), y, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(x2, xl, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# Layer stack pieces against PyTorch's library routines (float64, CPU).
# --------------------------------------------------------------------------
torch = pytest.importorskip("torch")


def test_layernorm_and_gate_match_library_routines():
    rng = _rng(41)
    H = 7
    x = rng.standard_normal((5, H)) * 3 + 1
    W = rng.standard_normal((H, H)) / np.sqrt(H)
    tx = torch.from_numpy(x)
    z_ref = torch.nn.functional.layer_norm(tx, (H,), eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.layernorm(x), z_ref, rtol=1e-12, atol=1e-12)
    h = torch.nn.functional.gelu(tx, approximate="none")
    out_ref = (h * torch.sigmoid(torch.nn.functional.linear(h, torch.from_numpy(W)))).numpy()
    np.testing.assert_allclose(oracle.gate(x, W), out_ref, rtol=1e-12, atol=1e-12)
    # W = 0: the gate is one half everywhere
    np.testing.assert_allclose(oracle.gate(x, np.zeros((H, H))), 0.5 * h.numpy(), rtol=1e-13)


def _tiny_stack(seed, B=2, L=8, H=3, P=2, nl=2):
    rng = _rng(seed)
    params = dict(
        **{"lambda": -rng.uniform(0.2, 0.8, (nl, P)) + 1j * rng.uniform(-4, 4, (nl, P))},
        log_dt=rng.uniform(np.log(0.01), np.log(0.5), (nl, P)),
        b_tilde=(rng.standard_normal((nl, P, H)) + 1j * rng.standard_normal((nl, P, H))) * 0.7,
        c_tilde=(rng.standard_normal((nl, H, P)) + 1j * rng.standard_normal((nl, H, P))) * 0.7,
        d=rng.standard_normal((nl, H)),
        W=rng.standard_normal((nl, H, H)) / np.sqrt(H),
    )
    u0 = rng.standard_normal((B, L, H))
    G = rng.standard_normal((B, L, H))
    return params, u0, G


def test_stack_forward_matches_composition_of_library_routines():
    params, u0, _ = _tiny_stack(51)
    u = u0.copy()
    H = u.shape[-1]
    for l in range(params["d"].shape[0]):
        z = torch.nn.functional.layer_norm(torch.from_numpy(u), (H,), eps=1e-5).numpy()
        dt = np.exp(params["log_dt"][l])
        lam = params["lambda"][l]
        gain = np.array([_ode_step(lam[p], 1.0, 0.0, dt[p]) for p in range(len(lam))])
        y = _lfilter_full_spectrum(np.exp(lam * dt), gain[:, None] * params["b_tilde"][l],
                                   params["c_tilde"][l], params["d"][l], z)
        h = torch.nn.functional.gelu(torch.from_numpy(y), approximate="none")
        o = h * torch.sigmoid(torch.nn.functional.linear(h, torch.from_numpy(params["W"][l])))
        u = u + o.numpy()
    np.testing.assert_allclose(oracle.stack(params, u0), u, rtol=1e-8, atol=1e-9)


def test_stack_backward_matches_central_finite_differences():
    """Gradients of L = sum(G * u_out), checked entry by entry (real and
    imaginary parts separately) with central differences, step 1e-6."""
    params, u0, G = _tiny_stack(52)
    _, gr = oracle.stack(params, u0, G)
    eps = 1e-6

    def loss(p, u):
        return float(np.sum(G * oracle.stack(p, u)))

    def check(name, grad, is_input=False):
        base = u0 if is_input else params[name]
        flat_grad = grad.reshape(-1)
        worst = 0.0
        for i in range(base.size):
            for part in ((1.0,) if not np.iscomplexobj(base) else (1.0, 1j)):
                def shifted(s):
                    arr = base.copy().reshape(-1)
                    arr[i] = arr[i] + s * eps * part
                    arr = arr.reshape(base.shape)
                    if is_input:
                        return loss(params, arr)
                    q = dict(params)
                    q[name] = arr
                    return loss(q, u0)
                fd = (shifted(1) - shifted(-1)) / (2 * eps)
                an = flat_grad[i].real if part == 1.0 else flat_grad[i].imag
                err = abs(fd - an) / max(1.0, abs(an))
                worst = max(worst, err)
        assert worst < 1e-6, (name, worst)

    check("u0", gr["du0"], is_input=True)
    check("lambda", gr["dlambda"])
    check("log_dt", gr["dlog_dt"])
    check("b_tilde", gr["db_tilde"])
    check("c_tilde", gr["dc_tilde"])
    check("d", gr["dd"])
    check("W", gr["dW"])
