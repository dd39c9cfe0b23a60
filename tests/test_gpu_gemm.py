"""GPU checks of the stack's dense contraction s5_gemm_bf16 (tcgen05 tensor
cores with TMA-fed operands, or the CUDA-core kernel for pitches TMA cannot
address) against float64 products of the same bf16-rounded operands.  Bar:
relative L2 error <= 1e-5 (exact bf16 products, fp32 accumulation)."""
import numpy as np
import pytest
import torch

from diagonal_state_space_gb300 import _native

from _parity import check

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _operand(rng, rows, cols, pitch):
    """bf16 [rows][cols] stored with row pitch `pitch`; returns (device
    tensor, float64 copy of the values)."""
    full = torch.zeros((rows, pitch), dtype=torch.bfloat16)
    vals = torch.from_numpy(rng.standard_normal((rows, cols)).astype(np.float32)).to(torch.bfloat16)
    full[:, :cols] = vals
    return full.cuda(), vals.double().numpy()


def _gemm(ta, tb, M, N, K, pad=0, seed=0):
    rng = np.random.default_rng(seed)
    # A: [M][K] or [K][M]; B: [K][N] or [N][K]
    a_rows, a_cols = (K, M) if ta else (M, K)
    b_rows, b_cols = (N, K) if tb else (K, N)
    A, a = _operand(rng, a_rows, a_cols, a_cols + pad)
    B, b = _operand(rng, b_rows, b_cols, b_cols + pad)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    lib = _native.lib()
    code = lib.s5_gemm_bf16(int(ta), int(tb), M, N, K, A.data_ptr(), a_cols + pad, B.data_ptr(), b_cols + pad,
                            C.data_ptr(), N, None)
    _native.check("s5_gemm_bf16", code)
    torch.cuda.synchronize()
    assert lib.s5_gemm_fault() == 0
    ref = (a.T if ta else a) @ (b.T if tb else b)
    return C.cpu().numpy().astype(np.float64), ref


@pytest.mark.parametrize("ta", [False, True])
@pytest.mark.parametrize("tb", [False, True])
@pytest.mark.parametrize("M,N,K", [(1, 64, 16), (130, 200, 72), (256, 512, 512), (300, 96, 1000)])
def test_gemm_matches_float64(ta, tb, M, N, K):
    got, ref = _gemm(ta, tb, M, N, K, seed=M + N + K)
    check(got, ref, TOL, "C")


@pytest.mark.parametrize("ta,tb", [(True, False), (False, True)])
def test_gemm_split_k(ta, tb):
    # few output tiles and a long K: K is split over the SMs and the partial
    # products are added into C
    got, ref = _gemm(ta, tb, 256, 256, 8192, seed=7)
    check(got, ref, TOL, "C")


@pytest.mark.parametrize("ta,tb", [(False, False), (True, True)])
def test_gemm_pitch_tma_cannot_address(ta, tb):
    # a row pitch of 30 bf16 (60 bytes) runs on the CUDA-core kernel
    got, ref = _gemm(ta, tb, 70, 30, 30, seed=3)
    check(got, ref, TOL, "C")
    got, ref = _gemm(ta, tb, 64, 64, 64, pad=2, seed=4)
    check(got, ref, TOL, "C")


def test_gemm_k_zero_writes_zeros():
    C = torch.full((5, 7), 3.0, dtype=torch.float32, device="cuda")
    x = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    code = _native.lib().s5_gemm_bf16(0, 0, 5, 7, 0, x.data_ptr(), 8, x.data_ptr(), 8, C.data_ptr(), 7, None)
    _native.check("s5_gemm_bf16", code)
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0


@pytest.mark.parametrize("K", [192, 8192])
def test_gemm_output_pitch_tma_cannot_store(K):
    # operands TMA can read, but an output pitch of N + 1 floats (not a
    # multiple of 16 bytes): the tensor-core kernel writes C with per-thread
    # stores (K = 8192 also splits K and adds the partial products atomically);
    # the padding column stays untouched
    rng = np.random.default_rng(K)
    M, N = 256, 64
    A, a = _operand(rng, M, K, K)
    B, b = _operand(rng, N, K, K)
    C = torch.full((M, N + 1), 7.0, dtype=torch.float32, device="cuda")
    lib = _native.lib()
    code = lib.s5_gemm_bf16(0, 1, M, N, K, A.data_ptr(), K, B.data_ptr(), K, C.data_ptr(), N + 1, None)
    _native.check("s5_gemm_bf16", code)
    torch.cuda.synchronize()
    assert lib.s5_gemm_fault() == 0
    got = C.cpu().numpy().astype(np.float64)
    check(got[:, :N], a @ b.T, TOL, "C")
    assert np.all(got[:, N] == 7.0)
