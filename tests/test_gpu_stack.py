"""GPU parity of the layer stack (pre-LayerNorm -> S5 layer -> gated
activation -> residual, forward and backward) against the float64 oracle.
Bar: relative L2 error <= 2e-2 per tensor (bf16 GEMM operands, complex fp32
scans); LayerNorm alone (fp32) <= 1e-5."""
import numpy as np
import pytest
import torch

import oracle
from diagonal_state_space_gb300 import stack as s5stack
from diagonal_state_space_gb300.workloads import make_stack_inputs

from _parity import dev, check

pytestmark = pytest.mark.gpu
BF16_TOL = 2e-2
GRADS = ["du0", "dlambda", "dlog_dt", "db_tilde", "dc_tilde", "dd", "dW"]


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _oracle_params(params, seqs=None):
    p = dict(params)
    p["lambda"] = p.pop("lambda_")
    return p


def _host(t):
    return t.detach().cpu().numpy()


@pytest.mark.parametrize("N,H", [(1, 1), (9, 100), (333, 200), (64, 512), (7, 130), (17, 1024)])
def test_layernorm_matches_oracle(N, H):
    rng = np.random.default_rng(N + H)
    x = (rng.standard_normal((N, H)) * 3 + 1.5).astype(np.float32)
    z16 = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
    z = s5stack.layernorm(dev(x), z_bf16=z16)
    oz = oracle.layernorm(x)
    check(_host(z), oz, 1e-5, "_host(z)")
    assert torch.equal(z16, z.to(torch.bfloat16))


@pytest.mark.parametrize("B,L,H,P,nl", [(1, 1, 32, 16, 1), (2, 77, 64, 32, 2), (3, 130, 48, 40, 2),
                                        (2, 257, 128, 64, 3), (2, 66, 30, 20, 1), (1, 200, 256, 96, 2)])
def test_stack_forward_backward_matches_oracle(B, L, H, P, nl):
    inp = make_stack_inputs(B, L, H, P, nl, seed=97 * B + L)
    st = s5stack.S5Stack(inp["params"], B, L)
    u = st.forward(dev(inp["u0"]))
    g = st.backward(dev(inp["G"]))
    torch.cuda.synchronize()
    ou, og = oracle.stack(_oracle_params(inp["params"]), inp["u0"], inp["G"])
    check(_host(u), ou, BF16_TOL, "_host(u)")
    for k in GRADS:
        check(_host(g[k]), og[k], BF16_TOL, k)


def test_stack_full_size_sampled_sequence():
    """The deep-stack workload at full size (B=32, L=1024, H=512, P=256, 6
    layers); the loss weights only sequence 0, so every parameter gradient
    and du0[0] equal the oracle's on that sequence alone, and du0 of the other
    sequences is exactly zero."""
    B, L, H, P, nl = 32, 1024, 512, 256, 6
    inp = make_stack_inputs(B, L, H, P, nl, seed=4000)
    G = np.zeros_like(inp["G"])
    G[0] = inp["G"][0]
    st = s5stack.S5Stack(inp["params"], B, L)
    u = st.forward(dev(inp["u0"]))
    u0_host = _host(u[0])
    g = st.backward(dev(G))
    torch.cuda.synchronize()
    ou, og = oracle.stack(_oracle_params(inp["params"]), inp["u0"][:1], G[:1])
    check(u0_host, ou[0], BF16_TOL, "u0_host")
    du0 = _host(g["du0"])
    check(du0[:1], og["du0"], BF16_TOL, "du0[:1]")
    assert not np.any(du0[1:])
    for k in GRADS[1:]:
        check(_host(g[k]), og[k], BF16_TOL, k)


def test_stack_rejects_misaligned_and_oversize():
    from diagonal_state_space_gb300 import _native
    lib = _native.lib()
    x = torch.zeros(64 + 1, dtype=torch.float32, device="cuda")
    z = torch.zeros(64, dtype=torch.float32, device="cuda")
    # misaligned input
    assert lib.s5_layernorm(x.data_ptr() + 4, z.data_ptr(), None, 1, 64, None) == 1
    # H beyond the register-resident row
    assert lib.s5_layernorm(x.data_ptr(), z.data_ptr(), None, 1, 2048, None) == 2


def _gate_inputs(N, H, seed, with_d=True):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    d = f(H) if with_d else np.zeros(H, np.float32)
    return dict(y_ssm=f(N, H), z=f(N, H), d=d, W=(f(H, H) / np.sqrt(H)).astype(np.float32), u=f(N, H),
                ubar=f(N, H))


def _gate_forward(inp):
    """s5_gate_residual on the device: (y, a, u_next) as torch tensors."""
    from diagonal_state_space_gb300 import _native
    lib = _native.lib()
    N, H = inp["u"].shape
    e = lambda *s, dt=torch.float32: torch.empty(s, dtype=dt, device="cuda")
    # the bf16 image of W through the library's own weight pass (P = 1 dummies)
    bb, ct, Wd = dev(np.zeros((1, H), np.complex64)), dev(np.zeros((H, 1), np.complex64)), dev(inp["W"])
    bs, cp, cx = e(2, H, dt=torch.bfloat16), e(H, 2, dt=torch.bfloat16), e(H, 2, dt=torch.bfloat16)
    w16 = e(H, H, dt=torch.bfloat16)
    assert lib.s5_stack_weights(bb.data_ptr(), ct.data_ptr(), Wd.data_ptr(), H, 1,
                                bs.data_ptr(), cp.data_ptr(), cx.data_ptr(), w16.data_ptr(), None) == 0
    y, a, un = e(N, H), e(N, H), e(N, H)
    ws = e(2 * N * H + 256, dt=torch.uint8)
    ys, z, d, u = dev(inp["y_ssm"]), dev(inp["z"]), dev(inp["d"]), dev(inp["u"])
    assert lib.s5_gate_residual(ys.data_ptr(), z.data_ptr(), d.data_ptr(), w16.data_ptr(), u.data_ptr(), N, H,
                                y.data_ptr(), a.data_ptr(), un.data_ptr(), ws.data_ptr(), ws.numel(), None) == 0
    return y, a, un, w16


# H a multiple of 8: W h on the tensor-core GEMM (one and two 256-column
# tiles, ragged rows and columns); 36 and 30: the CUDA-core GEMM (pitches TMA
# cannot address) and ragged elementwise tails
GATE_SHAPES = [(333, 64), (130, 48), (1000, 512), (77, 36), (50, 30)]


@pytest.mark.parametrize("N,H", GATE_SHAPES)
def test_gate_residual_matches_oracle(N, H):
    """u_next = u + GELU(y) sigmoid(W GELU(y)) with y = y_ssm + d z, against
    the oracle's gate (h and W are bf16 GEMM operands on the device)."""
    inp = _gate_inputs(N, H, seed=11 * N + H)
    y, a, un, _ = _gate_forward(inp)
    torch.cuda.synchronize()
    y_ref = inp["y_ssm"].astype(np.float64) + inp["d"].astype(np.float64) * inp["z"]
    check(_host(y), y_ref, 1e-6, "y")
    gate_ref = oracle.gate(y_ref, inp["W"])
    check(_host(un) - inp["u"], gate_ref, BF16_TOL, "u_next - u")


def _fd_rows(y, W, ubar, rows, eps=1e-5):
    """dL/dy on the given rows by central differences of the oracle's gate,
    L = sum(ubar * gate(y, W)); the gate acts on each row alone."""
    out = np.empty((len(rows), y.shape[1]))
    for i, r in enumerate(rows):
        yr = y[r:r + 1].astype(np.float64)
        for j in range(y.shape[1]):
            hp, hm = yr.copy(), yr.copy()
            h = eps * max(1.0, abs(yr[0, j]))
            hp[0, j] += h
            hm[0, j] -= h
            out[i, j] = (np.sum(ubar[r] * oracle.gate(hp, W)) - np.sum(ubar[r] * oracle.gate(hm, W))) / (2 * h)
    return out


@pytest.mark.parametrize("N,H", GATE_SHAPES)
def test_gate_backward_matches_oracle_differences(N, H):
    """ybar = dL/dy of L = sum(ubar * gate(y, W)) from s5_gate_backward (the
    kept y and a of s5_gate_residual) against central differences of the
    oracle's gate on sampled rows (first, middle, last), fp32 and bf16
    copies; dW on sampled entries against differences in W.  d = 0, so the
    kept y is y_ssm itself and the oracle sees the seeded values."""
    from diagonal_state_space_gb300 import _native
    lib = _native.lib()
    inp = _gate_inputs(N, H, seed=13 * N + H, with_d=False)
    y, a, _, w16 = _gate_forward(inp)
    e = lambda *s, dt=torch.float32: torch.empty(s, dtype=dt, device="cuda")
    ybar, ybar16, dW = e(N, H), e(N, H, dt=torch.bfloat16), e(H, H)
    ws = e(12 * N * H + 1024, dt=torch.uint8)
    ub = dev(inp["ubar"])
    assert lib.s5_gate_backward(ub.data_ptr(), y.data_ptr(), a.data_ptr(), w16.data_ptr(), N, H, ybar.data_ptr(),
                                ybar16.data_ptr(), dW.data_ptr(), ws.data_ptr(), ws.numel(), None) == 0
    torch.cuda.synchronize()
    yh = inp["y_ssm"].astype(np.float64)
    rows = sorted({0, N // 2, N - 1})
    ref = _fd_rows(yh, inp["W"], inp["ubar"].astype(np.float64), rows)
    got = _host(ybar)
    check(got[rows], ref, BF16_TOL, "ybar rows")
    assert torch.equal(ybar16, ybar.to(torch.bfloat16))
    # dW entries: L(W) over all rows, differences in one entry at a time
    rng = np.random.default_rng(N + H)
    ent = [(int(i), int(j)) for i, j in zip(rng.integers(0, H, 12), rng.integers(0, H, 12))]
    W0 = inp["W"].astype(np.float64)
    ubh = inp["ubar"].astype(np.float64)
    dref = []
    for i, j in ent:
        h = 1e-5
        Wp, Wm = W0.copy(), W0.copy()
        Wp[i, j] += h
        Wm[i, j] -= h
        dref.append((np.sum(ubh * oracle.gate(yh, Wp)) - np.sum(ubh * oracle.gate(yh, Wm))) / (2 * h))
    dW_h = _host(dW)
    check(np.array([dW_h[i, j] for i, j in ent]), np.array(dref), BF16_TOL, "dW entries")
