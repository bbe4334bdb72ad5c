"""fp64 reference ("oracle") of the owner-side Muon update of one 2-D matrix.

TEST INFRASTRUCTURE ONLY: used by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline legs of ``bench.py``. Nothing in the product imports it.

What it computes, per matrix W (stored ``rows x cols``) with gradient G and
momentum M, following the owner-side step described in "DMuon: Efficient
Distributed Muon Training with Near-Adam Overhead" (gist.science technical
summary, section 1 "Probleemstelling": Newton-Schulz iterations applied to the
momentum-aggregated gradient of a weight matrix, built on the product X X^T;
section 2 "Efficiente Gram Newton-Schulz Iteratie": iterate in the m x m space
of the short side when m < n):

1. momentum:      M' = mu * M + G;  U = G + mu * M' (Nesterov) or U = M'
2. normalise:     X0 = U / (||U||_F + eps)
3. orientation:   if rows > cols iterate on X0^T, so X is always m x n, m <= n
4. Newton-Schulz: for each step k with coefficients (a_k, b_k, c_k):
                     A = X X^T,  B = b_k A + c_k A A,  X <- a_k X + B X
5. orientation back, then the update  W' = W - lr * sqrt(max(1, rows/cols)) * X

The pages never print steps 1, 2, 4 or 5 as formulas; the forms used here (the
SGD-style heavy-ball momentum with a Nesterov option, eps added to the norm,
the quintic with (a, b, c) = (3.4445, -4.7750, 2.0315) and the
sqrt(max(1, rows/cols)) scale) are the plainest reading of "Muon" that the rest
of the pages support; every such reading is listed in the design notes.

Everything is float64 with dense ``@`` products: no symmetry tricks, no
padding, no blocking, so each line can be checked against the definition by eye.

Parity pins (tests/test_oracle_pins.py): spectral invariant by SVD brute force,
diagonal/permutation inputs, transpose commutation, the output singular-value
band, closed forms for ns_steps 0 and 1, orthogonal, rank-1 and zero inputs,
and the closed form of the momentum recurrence.
"""

from __future__ import annotations

import math
from typing import Sequence

import numpy as np

#: The quintic Newton-Schulz coefficients (a, b, c) of the Muon iteration.
DEFAULT_COEFFS = (3.4445, -4.7750, 2.0315)


def _coeff_list(ns_steps: int, coeffs) -> list[tuple[float, float, float]]:
    """Expand coefficients to one (a, b, c) triple per Newton-Schulz step.

    ``coeffs`` is either one triple (used for every step) or a sequence of
    ``ns_steps`` triples.
    """
    c = np.asarray(coeffs, dtype=np.float64)
    if c.ndim == 1:
        if c.shape != (3,):
            raise ValueError("coeffs must be (a, b, c) or a list of such triples")
        return [tuple(c)] * ns_steps
    if c.shape != (ns_steps, 3):
        raise ValueError("per-step coeffs must have shape (ns_steps, 3)")
    return [tuple(row) for row in c]


def momentum_update(M: np.ndarray, G: np.ndarray, mu: float, nesterov: bool):
    """Heavy-ball momentum with an optional Nesterov look-ahead.

    Returns ``(M_new, U)`` with ``M_new = mu*M + G`` and ``U`` the matrix that
    is orthogonalised: ``G + mu*M_new`` with Nesterov, else ``M_new``.
    ("momentum-aggregated gradients", gist.science summary section 1.)
    """
    M = np.asarray(M, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    M_new = mu * M + G
    U = G + mu * M_new if nesterov else M_new
    return M_new, U


def frobenius_normalize(U: np.ndarray, eps: float) -> np.ndarray:
    """``X0 = U / (||U||_F + eps)`` (eps added to the norm, not to its square)."""
    U = np.asarray(U, dtype=np.float64)
    norm = math.sqrt(float(np.sum(U * U)))
    return U / (norm + eps)


def newton_schulz(X: np.ndarray, coeff_steps: Sequence[tuple[float, float, float]]) -> np.ndarray:
    """Quintic Newton-Schulz on an ``m x n`` matrix, applied as written.

    Each step forms the Gram matrix ``A = X X^T`` (the product the gist.science
    summary, section 1, names as the reason NS needs the whole matrix), then
    ``B = b*A + c*A*A`` and ``X <- a*X + B*X``. The caller orients X so that
    the Gram matrix is formed on the short side.
    """
    X = np.asarray(X, dtype=np.float64)
    for a, b, c in coeff_steps:
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X


def newton_schulz_gram(X: np.ndarray, coeff_steps: Sequence[tuple[float, float, float]]) -> np.ndarray:
    """The same iteration carried out in the m x m Gram space.

    "DMuon: Efficient Distributed Muon Training with Near-Adam Overhead"
    (gist.science summary, section 2, "Gram Space Recurrence"): iterate on
    G = X X^T instead of the m x n matrix when m < n. The pages do not print
    the recurrence; this is the plain derivation from the quintic step. Each
    step maps X to P X with P = a I + b G + c G^2 a polynomial in G, so
    X_k = Q_k X_0 with Q_0 = I, Q_{k+1} = P_k Q_k, and G_{k+1} = P_k G_k P_k.
    Only the last step touches the m x n matrix again: X_S = Q_S X_0.
    """
    X0 = np.asarray(X, dtype=np.float64)
    m = X0.shape[0]
    I = np.eye(m)
    G = X0 @ X0.T
    Q = I
    for a, b, c in coeff_steps:
        P = a * I + b * G + c * (G @ G)
        Q = P @ Q
        G = P @ G @ P
    return Q @ X0


def orthogonalize(U: np.ndarray, ns_steps: int, coeffs=DEFAULT_COEFFS, eps: float = 1e-7) -> np.ndarray:
    """Normalise ``U``, run ``ns_steps`` Newton-Schulz steps on the short side,
    and return the result in ``U``'s orientation.

    "Short side": when rows > cols the iteration runs on the transpose, so the
    Gram matrix is ``min(rows, cols)`` square (gist.science summary section 2,
    m x m Gram space when m < n).
    """
    X = frobenius_normalize(U, eps)
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    X = newton_schulz(X, _coeff_list(ns_steps, coeffs))
    if transposed:
        X = X.T
    return X


def update_scale(rows: int, cols: int) -> float:
    """Shape-dependent step multiplier ``sqrt(max(1, rows/cols))``; rows is dim 0."""
    return math.sqrt(max(1.0, rows / cols))


def muon_step(W, G, M, *, lr: float, mu: float, nesterov: bool, ns_steps: int,
              coeffs=DEFAULT_COEFFS, eps: float = 1e-7):
    """One owner-side Muon step on one matrix (all in float64).

    Returns ``(W_new, M_new, X)``: the updated weight, the new momentum and the
    orthogonalised update X (before lr and the shape scale), each as float64 in
    the stored ``rows x cols`` orientation. ("The owner keeps the optimizer
    state and runs the Muon update (the Newton-Schulz iteration) exactly once
    per matrix": gist.science summary section 2.1, owner-centric execution.)
    """
    W = np.asarray(W, dtype=np.float64)
    M_new, U = momentum_update(M, G, mu, nesterov)
    X = orthogonalize(U, ns_steps, coeffs, eps)
    rows, cols = W.shape
    W_new = W - lr * update_scale(rows, cols) * X
    return W_new, M_new, X


# --------------------------------------------------------------------------
# storage rounding (round-to-nearest-even), used to compare against weights
# that the GPU stores in a narrower type
# --------------------------------------------------------------------------

_BF16_MAX = float.fromhex("0x1.fep127")


def _round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits: write x = f * 2**e with f in [0.5, 1),
    round f*256 to an integer with ties to even, and scale back. Values below
    the smallest normal (2**-126) round on the fixed grid 2**-133; values that
    round above the largest finite bfloat16 become inf.
    """
    x = np.asarray(x, dtype=np.float64)
    f, e = np.frexp(x)
    small = np.abs(x) < 2.0 ** -126
    r = np.ldexp(np.round(f * 256.0), e - 8)
    sub = np.round(np.ldexp(x, 133)) * 2.0 ** -133
    r = np.where(small, sub, r)
    with np.errstate(invalid="ignore"):
        big = np.abs(r) > _BF16_MAX
    r = np.where(big & np.isfinite(x), np.copysign(np.inf, x), r)
    return r


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round to the storage type ``"bf16"`` or ``"f32"`` (RNE), returned as float64."""
    if dtype == "bf16":
        return _round_bf16(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")

