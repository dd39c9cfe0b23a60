"""HiPPO-N initialisation of the S5 parameters (host side, numpy).

Sources: the review "S5: Simplified State Space Layers for Sequence Modeling",
"Initialization is part of the method" and "Paper equations beside executable
Python" row 5; the summary "SIMPLIFIED STATE SPACE LAYERS ...", App. B.1.1
(HiPPO-N as the normal part of HiPPO-LegS, block-diagonal variant) and
App. B.1.2 (B~ = V^-1 B, C~ = C V); the S4 page, "Diagonal plus low-rank"
(the spectrum -1/2 + i omega and its values at N = 8).

The initialiser runs once on the host, before any layer exists, and needs an
eigensolver; it is not on the layer's device path.
"""
from __future__ import annotations

import numpy as np


def hippo_normal(n: int) -> np.ndarray:
    """HiPPO-N = HiPPO-LegS + p p^T with p_k = sqrt(k + 1/2) (zero-based):
    -1/2 on the diagonal and the skew-symmetric entries
    sign(k - n) sqrt((n + 1/2)(k + 1/2)) off it (positive above the diagonal)."""
    if n < 1:
        raise ValueError("state size must be positive")
    idx = np.arange(n, dtype=np.float64) + 0.5
    a = np.sqrt(np.outer(idx, idx))
    a = np.triu(a, 1) - np.tril(a, -1)
    np.fill_diagonal(a, -0.5)
    return a


def hippo_normal_eig(n: int):
    """Eigen-decomposition of HiPPO-N: (eigenvalues [n] complex, V [n,n] unitary)
    with A = V diag(eigenvalues) V^H.  A = -1/2 I + S with S real
    skew-symmetric, so -iS is Hermitian; its eigenvalues omega give
    -1/2 + i omega, sorted by omega ascending."""
    a = hippo_normal(n)
    s = a + 0.5 * np.eye(n)
    omega, v = np.linalg.eigh(-1j * s)
    return -0.5 + 1j * omega, v


def init_s5(P: int, H: int, blocks: int = 1, dt_min: float = 1e-3, dt_max: float = 1e-1, seed: int = 0):
    """Parameters of one S5 layer with P stored complex modes:
    (lambda [P] complex, log_dt [P], b_tilde [P,H] complex, c_tilde [H,P]
    complex, d [H]).

    The state matrix is block-diagonal with `blocks` HiPPO-N blocks of size
    2P / blocks (summary App. B.1.1; blocks = 1 is the default single block).
    Each block's spectrum has conjugate pairs -1/2 +- i omega; one member of
    each pair is kept (the eigenvalues with omega >= 0 in ascending order),
    which is what "P stored modes" means.  B (2P x H) and C (H x 2P) are drawn
    densely (normal with variance 1/H and 1/(2P)) and moved into the eigenbasis,
    B~ = V^H B and C~ = C V (V unitary, so V^-1 = V^H), keeping the rows /
    columns of the stored modes.  log Delta ~ U[log dt_min, log dt_max)
    (App. B.1.2-3).  D ~ N(0, 1).
    """
    n = 2 * P
    if blocks < 1 or n % blocks:
        raise ValueError("2P must be a multiple of blocks")
    r = n // blocks
    lam_b, v_b = hippo_normal_eig(r)
    keep = np.nonzero(lam_b.imag >= 0)[0]
    if len(keep) != r // 2:
        keep = np.argsort(lam_b.imag)[r // 2:]
    rng = np.random.default_rng(seed)
    b_full = rng.standard_normal((n, H)) / np.sqrt(H)
    c_full = rng.standard_normal((H, n)) / np.sqrt(n)
    lam, bt, ct = [], [], []
    for j in range(blocks):
        sl = slice(j * r, (j + 1) * r)
        vb = v_b
        lam.append(lam_b[keep])
        bt.append((vb.conj().T @ b_full[sl])[keep])
        ct.append((c_full[:, sl] @ vb)[:, keep])
    lam = np.concatenate(lam)
    b_tilde = np.concatenate(bt, axis=0)
    c_tilde = np.concatenate(ct, axis=1)
    log_dt = rng.uniform(np.log(dt_min), np.log(dt_max), size=P)
    d = rng.standard_normal(H)
    return (lam.astype(np.complex64), log_dt.astype(np.float32), b_tilde.astype(np.complex64),
            c_tilde.astype(np.complex64), d.astype(np.float32))


__all__ = ["hippo_normal", "hippo_normal_eig", "init_s5"]
