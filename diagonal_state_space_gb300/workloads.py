"""Seeded synthetic inputs for the S5 layer workloads.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests; it therefore holds no arithmetic of the method itself -- only random
draws, the fixed initial spectrum and storage conversions (fp32 -> bf16 with
round-to-nearest-even).

Generators (the S5 paper's initialisation as summarised on the pages:
"SIMPLIFIED STATE SPACE LAYERS FOR SEQUENCE MODELING", App. B.1.2-B.1.3):
  u ~ N(0, 1)                              [B, L, H]
  lambda_n = -1/2 + i*pi*n, n = 0..P-1     (real part -1/2 as in HiPPO-N)
  log_dt ~ U[log 1e-3, log 1e-1)           [P]
  B~, C~: real and imaginary parts ~ N(0, 1/(2H))
  D ~ N(0, 1)                              [H]
  g ~ Exponential(mean 1)                  [B, L]   (irregular sampling gaps)
  W ~ N(0, 1/H)                            [H, H]   (gate of the layer stack)
  G ~ N(0, 1)                              [B, L, H] (loss weights of the stack)

All draws use numpy's PCG64 generator in the order listed, so a (shape, seed)
pair names one input set on every machine.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    # finite values: bits + 0x8000 stays below 2^32, so uint32 arithmetic is exact
    out = (bits + (((bits >> 16) & 1) + 0x7FFF)) & np.uint32(0xFFFF0000)
    return out.view(np.float32).reshape(x.shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 storage of float32 values that are already bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16).reshape(x.shape)


@dataclass(frozen=True)
class Workload:
    """One synthetic S5 workload: shapes, storage types and seed."""
    name: str
    B: int
    L: int
    H: int
    P: int
    u_dtype: str = "f32"      # storage type of u and y: "f32" or "bf16"
    proj_dtype: str = "f32"   # input type of the two projections
    varying_dt: bool = False  # per-step interval g_k * Delta_n
    bidirectional: bool = False  # forward and backward scans, C~ [H, 2P]
    method: str = "zoh"       # discretisation: "zoh" or "bilinear"
    clip_re: float = 0.0      # clip_eigs threshold on Re(lambda) (0: none)
    dt_scale: float = 1.0     # sampling-rate factor on Delta (old rate / new rate)
    streaming: bool = False   # one token per sequence per call (the step API), L calls
    layers: int = 0           # > 0: layer stack (pre-LN, SSM, gate, residual)
    seed: int = 0
    notes: str = field(default="", compare=False)

    @property
    def tokens(self) -> int:
        return self.B * self.L


# The five workloads of the S5 hot path.  The long-sequence case uses the
# Path-X length (16384), the irregular case stands in for the pendulum
# regression's irregular sampling.
WORKLOADS = {
    "small": Workload("small", 1, 1024, 32, 32, seed=0,
                      notes="single layer, fp32"),
    "fp32": Workload("fp32", 16, 4096, 128, 64, seed=1000,
                     notes="single layer, fp32 throughout"),
    "pathx_bf16": Workload("pathx_bf16", 8, 16384, 128, 128, u_dtype="bf16",
                           proj_dtype="bf16", seed=2000,
                           notes="long sequence, bf16 u/y and projections, complex fp32 scan"),
    "pathx_bf16_bidir": Workload("pathx_bf16_bidir", 8, 16384, 128, 128, u_dtype="bf16",
                                 proj_dtype="bf16", bidirectional=True, seed=2000,
                                 notes="the long-sequence shapes through the bidirectional layer"),
    "pathx_bf16_bilinear": Workload("pathx_bf16_bilinear", 8, 16384, 128, 128, u_dtype="bf16",
                                    proj_dtype="bf16", method="bilinear", clip_re=-1e-4,
                                    dt_scale=0.5, seed=2000,
                                    notes="the long-sequence shapes, bilinear discretisation with "
                                          "clip_eigs and a doubled sampling rate"),
    "stream": Workload("stream", 8, 1024, 128, 128, streaming=True, seed=4000,
                       notes="streaming inference: 8 sequences, 1024 single-token steps, fp32"),
    "irregular": Workload("irregular", 32, 2048, 256, 128, varying_dt=True, seed=3000,
                          notes="per-step interval g_k*Delta_n, fp32"),
    "stack6": Workload("stack6", 32, 1024, 512, 256, u_dtype="f32", proj_dtype="bf16",
                       layers=6, seed=4000,
                       notes="6 layers, pre-LN -> SSM -> gate -> residual, fwd + bwd"),
}


def spectrum(P: int) -> np.ndarray:
    """lambda_n = -1/2 + i*pi*n, stored as complex64."""
    n = np.arange(P, dtype=np.float64)
    return (-0.5 + 1j * np.pi * n).astype(np.complex64)


def _cnormal(rng, shape, var):
    std = np.float32(np.sqrt(var))
    re = rng.standard_normal(shape, dtype=np.float32) * std
    im = rng.standard_normal(shape, dtype=np.float32) * std
    return (re + 1j * im).astype(np.complex64)


def layer_params(rng, H: int, P: int) -> dict:
    """lambda, log_dt, B~, C~, D in the fixed draw order."""
    lam = spectrum(P)
    log_dt = rng.uniform(np.log(1e-3), np.log(1e-1), P).astype(np.float32)
    b_tilde = _cnormal(rng, (P, H), 1.0 / (2 * H))
    c_tilde = _cnormal(rng, (H, P), 1.0 / (2 * H))
    d = rng.standard_normal(H, dtype=np.float32)
    return dict(lambda_=lam, log_dt=log_dt, b_tilde=b_tilde, c_tilde=c_tilde, d=d)


def make_layer_inputs(B: int, L: int, H: int, P: int, seed: int, u_dtype: str = "f32",
                      varying_dt: bool = False, bidirectional: bool = False) -> dict:
    """Inputs of one S5 layer.  Keys: u (float32 values; bf16-representable when
    u_dtype == "bf16"), lambda_ (complex64 [P]), log_dt, b_tilde, c_tilde, d and,
    for irregular sampling, g [B, L]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    u = rng.standard_normal((B, L, H), dtype=np.float32)
    if u_dtype == "bf16":
        u = bf16_round(u)
    out = dict(u=u)
    out.update(layer_params(rng, H, P))
    if varying_dt:
        out["g"] = rng.exponential(1.0, (B, L)).astype(np.float32)
    if bidirectional:
        # C~ of the backward modes: the same complex-normal generator, its own stream
        rb = np.random.Generator(np.random.PCG64(seed + 1))
        sc = np.float32(np.sqrt(1.0 / (2 * H)))
        cb = (rb.standard_normal((H, P), dtype=np.float32) * sc
              + 1j * rb.standard_normal((H, P), dtype=np.float32) * sc).astype(np.complex64)
        out["c_tilde2"] = np.ascontiguousarray(np.concatenate([out["c_tilde"], cb], axis=1))
    return out


def make_stack_inputs(B: int, L: int, H: int, P: int, layers: int, seed: int) -> dict:
    """Inputs of the layer stack: u0, G and per-layer stacked parameters."""
    rng = np.random.Generator(np.random.PCG64(seed))
    u0 = rng.standard_normal((B, L, H), dtype=np.float32)
    rg = np.random.Generator(np.random.PCG64(seed + 1))
    G = rg.standard_normal((B, L, H), dtype=np.float32)
    per = []
    for l in range(layers):
        rl = np.random.Generator(np.random.PCG64(seed + 10 + l))
        p = layer_params(rl, H, P)
        p["W"] = rl.standard_normal((H, H), dtype=np.float32) * np.float32(np.sqrt(1.0 / H))
        per.append(p)
    stacked = {k: np.stack([p[k] for p in per]) for k in per[0]}
    return dict(u0=u0, G=G, params=stacked)


def make_inputs(w: Workload, B: int | None = None) -> dict:
    """Inputs of a named workload (optionally with fewer sequences)."""
    Bn = w.B if B is None else B
    if w.layers:
        return make_stack_inputs(Bn, w.L, w.H, w.P, w.layers, w.seed)
    return make_layer_inputs(Bn, w.L, w.H, w.P, w.seed, w.u_dtype, w.varying_dt, w.bidirectional)
