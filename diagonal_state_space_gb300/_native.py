"""ctypes loader of libs5.so.  Loading fails loudly: there is no fallback."""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libs5.so")

S5_F32, S5_BF16 = 0, 1
S5_NOALLOC_SCRATCH_BYTES = 16 << 20   # include/s5.h
STATUS = {0: "S5_OK", 1: "S5_ERR_INVALID_ARGUMENT", 2: "S5_ERR_UNSUPPORTED", 3: "S5_ERR_CUDA",
          4: "S5_ERR_TIMEOUT", 5: "S5_ERR_NONFINITE"}

# Every exported entry point of include/s5.h: name -> (restype, argtypes)
_vp, _i, _sz, _ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong
SIGNATURES = {
    "s5_discretize": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp, _vp]),
    "s5_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp,
                        _vp, _sz, _vp]),
    "s5_forward_varying_dt": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i,
                                   _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "s5_forward_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _vp,
                                _vp, _vp]),
    "s5_workspace_size": (_sz, [_i, _i, _i, _i]),
    "s5_discretize_ex": (_i, [_vp, _vp, _vp, _i, _i, _i, ctypes.c_float, ctypes.c_float, _vp, _vp, _vp]),
    "s5_step": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp]),
    "s5_forward_bidirectional": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _vp, _sz, _vp]),
    "s5_bidirectional_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "s5_sync_status": (_i, [_vp, _vp]),
    "s5_status_string": (ctypes.c_char_p, [_i]),
    "s5_last_cuda_error": (ctypes.c_char_p, []),
    # layer stack
    "s5_stack_workspace_size": (_sz, [_i, _i, _i, _i]),
    "s5_stack_last_error": (ctypes.c_char_p, []),
    "s5_layernorm": (_i, [_vp, _vp, _vp, _ll, _i, _vp]),
    "s5_stack_weights": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "s5_ssm_forward_states": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp,
                                   _vp, _vp, _sz, _vp]),
    "s5_gate_residual": (_i, [_vp, _vp, _vp, _vp, _vp, _ll, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "s5_gate_backward": (_i, [_vp, _vp, _vp, _vp, _ll, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "s5_ssm_backward": (_i, [_vp] * 16 + [_i] * 4 + [_vp] * 7 + [_sz, _vp]),
    "s5_gemm_bf16": (_i, [_i, _i, _i, _i, _i, _vp, _ll, _vp, _ll, _vp, _ll, _vp]),
    "s5_gemm_fault": (_i, []),
}

_lock = threading.Lock()
_lib = None


class S5Error(RuntimeError):
    def __init__(self, fn: str, code: int, detail: str = ""):
        self.code = code
        msg = "%s failed: %s" % (fn, STATUS.get(code, str(code)))
        if detail:
            msg += " (%s)" % detail
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """The loaded libs5.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libs5.so is not built (%s); run __graft_entry__.build() or "
                                   "python diagonal_state_space_gb300/build.py" % LIB_PATH)
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(h, name)
                f.restype = res
                f.argtypes = args
            _lib = h
    return _lib


def check(fn: str, code: int) -> None:
    if code != 0:
        detail = ""
        if code == 3:
            getter = lib().s5_stack_last_error if fn in STACK_FUNCTIONS else lib().s5_last_cuda_error
            detail = getter().decode()
        raise S5Error(fn, code, detail)


STACK_FUNCTIONS = {"s5_layernorm", "s5_stack_weights", "s5_ssm_forward_states", "s5_gate_residual",
                   "s5_gate_backward", "s5_ssm_backward", "s5_gemm_bf16"}
