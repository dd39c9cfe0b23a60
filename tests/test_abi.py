"""CPU-only checks of the C ABI: the library loads, exports every entry point
that include/s5.h declares, and rejects bad arguments on the host without
touching the GPU."""
import ctypes
import os
import re

import pytest

from diagonal_state_space_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "s5.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(s5_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_native.LIB_PATH):
        from diagonal_state_space_gb300 import build
        build.build()
    return _native.lib()


def test_every_declared_entry_point_is_exported_and_bound(lib):
    names = _declared()
    assert "s5_forward" in names and "s5_discretize" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in _native.SIGNATURES, "binding lacks %s" % n
    assert set(_native.SIGNATURES) == set(names)


def test_status_strings(lib):
    for code in range(6):
        assert lib.s5_status_string(code)
    assert lib.s5_status_string(99) == b"unknown status"


def test_workspace_size(lib):
    assert lib.s5_workspace_size(1, 1024, 32, 32) > 256
    assert lib.s5_workspace_size(0, 0, 32, 32) >= 256
    assert lib.s5_workspace_size(-1, 1, 1, 1) == 0
    assert lib.s5_workspace_size(1, 1, 0, 1) == 0
    a = lib.s5_workspace_size(8, 16384, 128, 128)
    b = lib.s5_workspace_size(8, 2 * 16384, 128, 128)
    assert b > a


def test_host_validation_needs_no_gpu(lib):
    INV = 1
    fake = ctypes.c_void_p(1 << 20)          # aligned, never dereferenced on rejection
    mis = ctypes.c_void_p((1 << 20) + 4)     # misaligned
    assert lib.s5_discretize(None, fake, fake, 4, 4, fake, fake, None) == INV
    assert lib.s5_discretize(fake, fake, fake, 0, 4, fake, fake, None) == INV
    assert lib.s5_discretize(fake, mis, fake, 4, 4, fake, fake, None) == INV
    args = [fake, fake, fake, fake, fake, 0, fake, 0, 0, 2, 8, 4, 4, None, None, fake, 1 << 30, None]
    bad = list(args); bad[9] = -1                      # B < 0
    assert lib.s5_forward(*bad) == INV
    bad = list(args); bad[5] = 7                       # unknown dtype
    assert lib.s5_forward(*bad) == INV
    bad = list(args); bad[16] = 16                     # workspace too small
    assert lib.s5_forward(*bad) == INV
    bad = list(args); bad[4] = mis                     # misaligned u
    assert lib.s5_forward(*bad) == INV
    vargs = [fake, fake, fake, fake, fake, None, fake, 0, fake, 0, 0, 2, 8, 4, 4, None, None,
             fake, 1 << 30, None]
    assert lib.s5_forward_varying_dt(*vargs) == INV    # dt_scale missing
    assert lib.s5_sync_status(None, None) == INV


def test_host_validation_of_the_next_row_entry_points(lib):
    INV, OK = 1, 0
    fake = ctypes.c_void_p(1 << 20)          # aligned, never dereferenced on these paths
    mis = ctypes.c_void_p((1 << 20) + 4)
    f = ctypes.c_float
    # discretisation options: unknown method, non-positive rate factor, positive clip
    ok_args = [fake, fake, fake, 4, 4, 0, f(0.0), f(1.0), fake, fake, None]
    for i, v in ((5, 2), (7, f(0.0)), (7, f(-1.0)), (6, f(1e-4)), (3, 0)):
        bad = list(ok_args); bad[i] = v
        assert lib.s5_discretize_ex(*bad) == INV
    bad = list(ok_args); bad[1] = mis
    assert lib.s5_discretize_ex(*bad) == INV
    # streaming step: bad sizes and parameters are rejected; an empty batch is a no-op
    assert lib.s5_step(fake, fake, fake, fake, fake, fake, fake, -1, 8, 4, None) == INV
    assert lib.s5_step(None, fake, fake, fake, fake, fake, fake, 1, 8, 4, None) == INV
    assert lib.s5_step(fake, fake, fake, fake, fake, fake, fake, 1, 0, 4, None) == INV
    assert lib.s5_step(fake, fake, fake, fake, None, None, None, 0, 8, 4, None) == OK
    # bidirectional layer
    assert lib.s5_bidirectional_workspace_size(-1, 1, 1, 1, 0, 0) == 0
    assert lib.s5_bidirectional_workspace_size(1, 1, 1, 1, 9, 0) == 0
    n1 = lib.s5_bidirectional_workspace_size(2, 100, 8, 4, 0, 0)
    assert n1 >= lib.s5_workspace_size(2, 100, 8, 4)
    bargs = [fake, fake, fake, fake, fake, 0, fake, 0, 0, 2, 100, 8, 4, fake, n1, None]
    bad = list(bargs); bad[2] = None                   # no c_tilde2
    assert lib.s5_forward_bidirectional(*bad) == INV
    bad = list(bargs); bad[14] = 16                    # workspace too small
    assert lib.s5_forward_bidirectional(*bad) == INV
    bad = list(bargs); bad[10] = 0                     # L = 0: nothing to do
    assert lib.s5_forward_bidirectional(*bad) == OK


def test_host_validation_of_the_gemm(lib):
    INV = 1
    fake = ctypes.c_void_p(1 << 20)
    # negative sizes, missing operands, pitches below the row length
    assert lib.s5_gemm_bf16(0, 0, -1, 4, 4, fake, 4, fake, 4, fake, 4, None) == INV
    assert lib.s5_gemm_bf16(0, 0, 4, 4, 4, None, 4, fake, 4, fake, 4, None) == INV
    assert lib.s5_gemm_bf16(0, 0, 4, 4, 8, fake, 4, fake, 4, fake, 4, None) == INV   # lda < K
    assert lib.s5_gemm_bf16(1, 0, 8, 4, 4, fake, 4, fake, 4, fake, 4, None) == INV   # ta: lda < M
    assert lib.s5_gemm_bf16(0, 1, 4, 4, 8, fake, 8, fake, 4, fake, 4, None) == INV   # tb: ldb < K
    assert lib.s5_gemm_bf16(0, 0, 4, 8, 4, fake, 4, fake, 8, fake, 4, None) == INV   # ldc < N
    # an empty product is a no-op that launches nothing
    assert lib.s5_gemm_bf16(0, 0, 0, 4, 4, None, 0, None, 0, None, 0, None) == 0
