"""Layer stack: pre-LayerNorm -> S5 layer -> gated activation -> residual,
repeated over layers, with its backward.

Marshalling and buffer management only: every numeric step is a call into
libs5.so (``s5_discretize``, ``s5_stack_weights``, ``s5_layernorm``,
``s5_ssm_forward_states``, ``s5_gate_residual``, ``s5_gate_backward``,
``s5_ssm_backward``).  Tensors are torch CUDA tensors used as device buffers.

Layer l (review "S5: Simplified State Space Layers for Sequence Modeling",
row 4; paper section 6; wiki "Method" step 4):
    z = LayerNorm(u_l)   (no affine, eps 1e-5)
    y = S5(z)            (ZOH, complex fp32 scan, bf16 GEMM operands)
    u_{l+1} = u_l + GELU(y) * sigmoid(W GELU(y))
The loss of the backward is sum(G * u_out): ``backward(G)`` returns dL/du0 and
the parameter gradients, with grad(z) = dL/dRe z + i dL/dIm z for complex
parameters.
"""
from __future__ import annotations

import torch

from . import _native
from ._native import check

_C64, _F32, _BF16 = torch.complex64, torch.float32, torch.bfloat16


def _p(t):
    return None if t is None else t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


class S5Stack:
    """A stack of S5 layers on one GPU.

    params: dict of per-layer stacked tensors (or arrays) lambda_ [nl,P]
    complex64, log_dt [nl,P] f32, b_tilde [nl,P,H] complex64, c_tilde [nl,H,P]
    complex64, d [nl,H] f32, W [nl,H,H] f32.
    """

    def __init__(self, params: dict, B: int, L: int, device="cuda"):
        dev = torch.device(device)
        as_t = lambda a, dt: torch.as_tensor(a).to(device=dev, dtype=dt).contiguous()
        self.lam = as_t(params["lambda_"], _C64)
        self.log_dt = as_t(params["log_dt"], _F32)
        self.b_tilde = as_t(params["b_tilde"], _C64)
        self.c_tilde = as_t(params["c_tilde"], _C64)
        self.d = as_t(params["d"], _F32)
        self.W = as_t(params["W"], _F32)
        self.nl, self.P = self.lam.shape
        self.H = self.d.shape[1]
        self.B, self.L = B, L
        nl, P, H, T = self.nl, self.P, self.H, B * L
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
        # discretised parameters and bf16 GEMM operands
        self.lbar = e((nl, P), _C64)
        self.bbar = e((nl, P, H), _C64)
        self.bs = e((nl, 2 * P, H), _BF16)
        self.cp = e((nl, H, 2 * P), _BF16)
        self.cx = e((nl, H, 2 * P), _BF16)
        self.w16 = e((nl, H, H), _BF16)
        # activations kept for the backward
        self.u = e((nl + 1, B, L, H), _F32)
        self.z = e((nl, B, L, H), _F32)
        self.z16 = e((nl, B, L, H), _BF16)
        self.x = e((nl, B, L, P), _C64)
        self.X = e((nl, B, L, 2 * P), _BF16)
        self.y = e((nl, B, L, H), _F32)
        self.a = e((nl, B, L, H), _F32)
        self.yssm = e((B, L, H), _F32)
        # backward buffers
        self.ubar = e((B, L, H), _F32)
        self.ybar = e((B, L, H), _F32)
        self.ybar16 = e((B, L, H), _BF16)
        nbytes = int(_native.lib().s5_stack_workspace_size(B, L, H, P))
        if nbytes == 0:
            raise ValueError("invalid stack sizes")
        self.ws = e((nbytes,), torch.uint8)
        self.T = T

    # ------------------------------------------------------------------ forward
    def forward(self, u0) -> torch.Tensor:
        lib, st = _native.lib(), _stream()
        B, L, H, P, T = self.B, self.L, self.H, self.P, self.T
        self.u[0].copy_(torch.as_tensor(u0, dtype=_F32).reshape(B, L, H))
        # the zero-order hold acts per mode: all layers' modes in one call
        check("s5_discretize", lib.s5_discretize(
            _p(self.lam), _p(self.log_dt), _p(self.b_tilde), self.nl * P, H, _p(self.lbar),
            _p(self.bbar), st))
        for l in range(self.nl):
            check("s5_stack_weights", lib.s5_stack_weights(
                _p(self.bbar[l]), _p(self.c_tilde[l]), _p(self.W[l]), H, P, _p(self.bs[l]),
                _p(self.cp[l]), _p(self.cx[l]), _p(self.w16[l]), st))
            check("s5_layernorm", lib.s5_layernorm(_p(self.u[l]), _p(self.z[l]), _p(self.z16[l]),
                                                   T, H, st))
            check("s5_ssm_forward_states", lib.s5_ssm_forward_states(
                _p(self.lbar[l]), _p(self.bs[l]), _p(self.cp[l]), _p(self.d[l]), _p(self.z[l]),
                _p(self.z16[l]), B, L, H, P, None, _p(self.yssm), _p(self.x[l]), _p(self.X[l]),
                _p(self.ws), self.ws.numel(), st))
            check("s5_gate_residual", lib.s5_gate_residual(
                _p(self.yssm), _p(self.z[l]), _p(self.d[l]), _p(self.w16[l]), _p(self.u[l]), T, H,
                _p(self.y[l]), _p(self.a[l]), _p(self.u[l + 1]), _p(self.ws), self.ws.numel(), st))
        return self.u[self.nl]

    # ----------------------------------------------------------------- backward
    def backward(self, G) -> dict:
        """dL/d(inputs) for L = sum(G * u_out), after forward()."""
        lib, st = _native.lib(), _stream()
        B, L, H, P, T, nl = self.B, self.L, self.H, self.P, self.T, self.nl
        dev = self.u.device
        g = dict(dlambda=torch.empty((nl, P), dtype=_C64, device=dev),
                 dlog_dt=torch.empty((nl, P), dtype=_F32, device=dev),
                 db_tilde=torch.empty((nl, P, H), dtype=_C64, device=dev),
                 dc_tilde=torch.empty((nl, H, P), dtype=_C64, device=dev),
                 dd=torch.empty((nl, H), dtype=_F32, device=dev),
                 dW=torch.empty((nl, H, H), dtype=_F32, device=dev))
        self.ubar.copy_(torch.as_tensor(G, dtype=_F32).reshape(B, L, H))
        for l in range(nl - 1, -1, -1):
            check("s5_gate_backward", lib.s5_gate_backward(
                _p(self.ubar), _p(self.y[l]), _p(self.a[l]), _p(self.w16[l]), T, H, _p(self.ybar),
                _p(self.ybar16), _p(g["dW"][l]), _p(self.ws), self.ws.numel(), st))
            check("s5_ssm_backward", lib.s5_ssm_backward(
                _p(self.lam[l]), _p(self.log_dt[l]), _p(self.b_tilde[l]), _p(self.lbar[l]),
                _p(self.bs[l]), _p(self.cx[l]), _p(self.d[l]), _p(self.u[l]), _p(self.z[l]),
                _p(self.z16[l]), _p(self.x[l]), _p(self.X[l]), None, _p(self.ybar),
                _p(self.ybar16), _p(self.ubar), B, L, H, P, _p(self.ubar), _p(g["dlambda"][l]),
                _p(g["dlog_dt"][l]), _p(g["db_tilde"][l]), _p(g["dc_tilde"][l]), _p(g["dd"][l]),
                _p(self.ws), self.ws.numel(), st))
        g["du0"] = self.ubar
        return g


def layernorm(x, z=None, z_bf16=None):
    """LayerNorm without affine over the last axis (eps 1e-5) through
    s5_layernorm; returns z (and fills z_bf16 if given)."""
    H = x.shape[-1]
    if z is None:
        z = torch.empty_like(x)
    check("s5_layernorm", _native.lib().s5_layernorm(_p(x), _p(z), _p(z_bf16), x.numel() // H, H,
                                                     _stream()))
    return z


__all__ = ["S5Stack", "layernorm"]
