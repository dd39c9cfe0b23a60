"""s5_forward_noalloc: the forward entry point for callers that cannot
allocate device memory (for instance a plugin inside a host application that
owns all device memory).  It must give the same result as s5_forward with a
caller workspace, call after call, and refuse sizes beyond its fixed scratch.

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

from _parity import host, layer_to_device, rel_l2

pytestmark = pytest.mark.gpu

FP32_TOL = 1e-5


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


@pytest.mark.parametrize("B,L,H,P", [(1, 1024, 32, 32), (4, 3000, 64, 48), (8, 16384, 128, 128)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(B, L, H, P):
    inp = make_layer_inputs(B, L, H, P, seed=900 + B + P)
    t = layer_to_device(inp)
    lb, bb = api.s5_discretize(t["lam"], t["log_dt"], t["b_tilde"])
    x0 = torch.randn(B, P, dtype=torch.complex64, device="cuda")
    ref_y, ref_x = api.s5_forward(lb, bb, t["c_tilde"], t["d"], t["u"], x0=x0, x_last=True)
    for _ in range(2):
        y = torch.full_like(ref_y, float("nan"))
        xl = torch.full_like(ref_x, float("nan"))
        api.s5_forward_noalloc(lb, bb, t["c_tilde"], t["d"], t["u"], y, x0=x0, x_last=xl)
        torch.cuda.synchronize()
        assert rel_l2(host(y), host(ref_y)) <= FP32_TOL
        assert rel_l2(host(xl), host(ref_x)) <= FP32_TOL


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
