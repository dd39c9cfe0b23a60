"""s5_forward_noalloc: the forward entry point for callers that cannot
allocate device memory (for instance a plugin inside a host application that
owns all device memory).  It must match the oracle within the layer's
tolerances and give the result of s5_forward with a caller workspace, call
after call, and refuse sizes beyond its fixed scratch.

Kept in a file that pytest collects last, so that a run stopping at its first
failure has already run every other test; it also passes on its own in a
fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from diagonal_state_space_gb300 import _native, api
from diagonal_state_space_gb300.workloads import make_layer_inputs

from _parity import check, host, layer_to_device, oracle_forward

pytestmark = pytest.mark.gpu

FP32_TOL = 1e-5
BF16_TOL = 2e-2


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


# (B, L, H, P, u/y dtype, projection dtype): fp32 and bf16 CUDA-core cases,
# and bf16 at H = P = 128 (the tensor-core kernel), up to the long-sequence
# shape (B=8, L=16384).
CASES = [
    (1, 1024, 32, 32, "f32", "f32"),
    (4, 3000, 64, 48, "f32", "f32"),
    (8, 16384, 128, 128, "f32", "f32"),
    (4, 3000, 64, 48, "f32", "bf16"),
    (2, 2500, 64, 32, "bf16", "bf16"),
    (2, 4160, 128, 128, "bf16", "bf16"),
    (8, 16384, 128, 128, "bf16", "bf16"),
]


@pytest.mark.parametrize("B,L,H,P,io,proj", CASES)
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls(B, L, H, P, io, proj):
    inp = make_layer_inputs(B, L, H, P, seed=900 + B + P, u_dtype=io)
    rng = np.random.default_rng(901 + B)
    x0_np = (rng.standard_normal((B, P)) + 1j * rng.standard_normal((B, P))).astype(np.complex64)
    t = layer_to_device(inp, io)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    x0 = torch.from_numpy(x0_np).cuda()
    oy, oxl = oracle_forward(inp, x0=x0_np.astype(np.complex128))
    # x_last keeps a fraction |lambda_bar|^L of x0: its float64 reference is
    # the oracle on complex64 lambda_bar / B_bar (the stored parameters)
    _, oxl_c64 = oracle_forward(inp, x0=x0_np.astype(np.complex128), c64_params=True)
    tol = FP32_TOL if (io == "f32" and proj == "f32") else BF16_TOL
    ref_y, ref_x = api.s5_forward(lb, bb, t["c_tilde"], t["d"], t["u"], proj_dtype=proj, x0=x0,
                                  x_last=True)
    # two calls back to back on one stream, no synchronisation between them
    outs = []
    for _ in range(2):
        y = torch.full_like(ref_y, float("nan"))
        xl = torch.full_like(ref_x, float("nan"))
        api.s5_forward_noalloc(lb, bb, t["c_tilde"], t["d"], t["u"], y, proj_dtype=proj, x0=x0,
                               x_last=xl)
        outs.append((y, xl))
    torch.cuda.synchronize()
    for y, xl in outs:
        check(host(y), oy, tol, "y vs oracle (%s u/y, %s proj)" % (io, proj))
        check(host(xl), oxl_c64, tol, "x_last vs oracle (c64 params)")
        # the same kernels as s5_forward on a caller workspace; the look-back
        # may reach a carry through a tile's aggregate or its inclusive state,
        # so fp32 values can differ in their last bits and bf16 outputs by one
        # unit in the last place
        check(host(y), host(ref_y), 1e-6 if io == "f32" else 1e-4, "y vs s5_forward")
        check(host(xl), host(ref_x), 1e-6, "x_last vs s5_forward")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _native.lib()
    B, L, H, P = 64, 65536, 128, 128
    assert lib.s5_workspace_size(B, L, H, P) > _native.S5_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)        # aligned; never dereferenced when rejected
    code = lib.s5_forward_noalloc(fake, fake, fake, fake, fake, 0, fake, 0, 0, B, L, H, P,
                                  None, None, None)
    assert code == 1                        # S5_ERR_INVALID_ARGUMENT
    u = torch.empty(B, L, H, dtype=torch.float32, device="meta")
    with pytest.raises(api.S5Error, match="carry scratch"):
        api.s5_forward_noalloc(None, torch.empty(P, H), None, None, u, None)
