"""Pins for the fp64 oracle against facts the mathematics fixes (CPU only).

Newton-Schulz acts on singular values alone: with U = P diag(s) Q^T, each step
maps X = P diag(x) Q^T to P diag(p(x)) Q^T where p(x) = a x + b x^3 + c x^5
(because (X X^T) X = P diag(x^3) Q^T). So the whole iteration equals the scalar
map f = p_S o ... o p_1 applied to the normalised singular values. These tests
check the oracle's matrix iteration against that scalar map computed from an
SVD (numpy.linalg.svd), plus diagonal, permutation, transpose, band, closed
form, momentum and rounding facts. A dropped term, a swapped coefficient, a
transposed product or a wrong normalisation fails at least one of them.
"""

import math

import numpy as np
import pytest
import torch

from oracle import muon_ref as ref

A, B, C = 3.4445, -4.7750, 2.0315


def p_scalar(x, a=A, b=B, c=C):
    return a * x + b * x ** 3 + c * x ** 5


def f_scalar(x, steps, coeffs=None):
    coeffs = coeffs or [(A, B, C)] * steps
    for a, b, c in coeffs:
        x = p_scalar(x, a, b, c)
    return x


def spectral_expected(U, steps, eps=1e-7, coeffs=None):
    P, s, Qt = np.linalg.svd(U, full_matrices=False)
    s_hat = s / (np.linalg.norm(s) + eps)
    return (P * f_scalar(s_hat, steps, coeffs)) @ Qt


SHAPES = [(1, 5), (5, 1), (4, 4), (8, 16), (16, 8), (12, 12), (3, 7), (7, 3), (1, 1)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("steps", [0, 1, 2, 5])
def test_spectral_invariant_svd_brute_force(shape, steps):
    for seed in range(10):
        U = np.random.default_rng(seed).standard_normal(shape)
        got = ref.orthogonalize(U, steps)
        want = spectral_expected(U, steps)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-11)


def test_spectral_invariant_per_step_coeffs():
    coeffs = [(3.4445, -4.7750, 2.0315), (2.0, -1.5, 0.5), (1.875, -1.25, 0.375)]
    for seed in range(5):
        U = np.random.default_rng(100 + seed).standard_normal((6, 11))
        got = ref.orthogonalize(U, 3, coeffs)
        want = spectral_expected(U, 3, coeffs=coeffs)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-11)


def test_toy_config_against_svd():
    # the 4 fp32 matrices of the toy workload, checked one by one through the scalar map
    for i in range(4):
        U = np.random.default_rng(7 + i).standard_normal((128, 256)).astype(np.float32).astype(np.float64)
        got = ref.orthogonalize(U, 5)
        want = spectral_expected(U, 5)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-10)


def test_diagonal_stays_diagonal():
    d = np.array([3.0, -1.0, 0.5, 2.0, 1e-3, 0.0])
    U = np.zeros((6, 9))
    U[np.arange(6), np.arange(6)] = d
    got = ref.orthogonalize(U, 5)
    dh = d / (np.linalg.norm(d) + 1e-7)
    want = np.zeros_like(U)
    # p is odd, so the sign of each diagonal entry is kept
    want[np.arange(6), np.arange(6)] = f_scalar(dh, 5)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)
    off = got.copy()
    off[np.arange(6), np.arange(6)] = 0
    assert np.all(off == 0.0)


def test_permutation_of_diagonal():
    d = np.array([1.0, 2.0, 3.0, 4.0, 5.0])
    perm = np.array([3, 0, 4, 1, 2])
    Pm = np.eye(5)[perm]
    U = Pm @ np.diag(d)
    got = ref.orthogonalize(U, 5)
    want = Pm @ np.diag(f_scalar(d / (np.linalg.norm(d) + 1e-7), 5))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)


@pytest.mark.parametrize("shape", [(9, 4), (4, 9), (8, 8), (1, 6)])
def test_transpose_commutes(shape):
    U = np.random.default_rng(3).standard_normal(shape)
    a = ref.orthogonalize(U.T.copy(), 5)
    b = ref.orthogonalize(U, 5).T
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)


def test_output_band_on_gaussian_inputs():
    # Scalar facts of the quintic, evaluated on a 2M-point grid of [0, 1]:
    # max p = 1.2023686 (at x ~ 0.5545), and after 5 steps every input
    # singular value >= 1e-2 (of the normalised matrix) lands in
    # [0.6818314, 1.1343573].
    for shape in [(256, 1024), (128, 512), (512, 128)]:
        U = np.random.default_rng(11).standard_normal(shape)
        X = ref.orthogonalize(U, 5)
        s = np.linalg.svd(X, compute_uv=False)
        s_in = np.linalg.svd(U, compute_uv=False) / np.linalg.norm(U)
        assert s_in.min() >= 1e-2
        assert s.min() >= 0.6818314 - 1e-9 and s.max() <= 1.1343573 + 1e-9
        assert s.max() <= 1.2023687


def test_closed_form_zero_steps():
    U = np.random.default_rng(5).standard_normal((7, 13))
    np.testing.assert_allclose(ref.orthogonalize(U, 0), U / (math.sqrt((U * U).sum()) + 1e-7), rtol=1e-15, atol=0)


def test_closed_form_orthogonal_input():
    n = 16
    Q, _ = np.linalg.qr(np.random.default_rng(9).standard_normal((n, n)))
    alpha = 2.5
    X = ref.orthogonalize(alpha * Q, 5)
    # all singular values equal alpha, so the normalised ones are 1/sqrt(n) (eps aside)
    scale = f_scalar(alpha / (alpha * math.sqrt(n) + 1e-7), 5)
    np.testing.assert_allclose(X, scale * Q, rtol=0, atol=1e-13)


def test_closed_form_rank_one():
    u = np.random.default_rng(1).standard_normal(6)
    v = np.random.default_rng(2).standard_normal(10)
    U = np.outer(u, v)
    X = ref.orthogonalize(U, 5)
    nu = np.linalg.norm(u) * np.linalg.norm(v)
    want = f_scalar(nu / (nu + 1e-7), 5) * U / nu
    np.testing.assert_allclose(X, want, rtol=0, atol=1e-13)
    # f(1) after five quintic steps
    assert abs(f_scalar(1.0, 5) - 0.6964364094697522) < 1e-12


def test_zero_gradient_leaves_weight_unchanged():
    W = np.random.default_rng(0).standard_normal((5, 8))
    Z = np.zeros((5, 8))
    W2, M2, X = ref.muon_step(W, Z, Z, lr=0.02, mu=0.95, nesterov=True, ns_steps=5)
    assert np.all(X == 0) and np.all(M2 == 0) and np.array_equal(W2, W)


def test_momentum_recurrence_closed_form():
    rng = np.random.default_rng(4)
    mu = 0.9
    Gs = [rng.standard_normal((3, 4)) for _ in range(6)]
    M = np.zeros((3, 4))
    for k, G in enumerate(Gs, start=1):
        M, U = ref.momentum_update(M, G, mu, nesterov=True)
        closed = sum(mu ** (k - j) * Gs[j - 1] for j in range(1, k + 1))
        np.testing.assert_allclose(M, closed, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(U, G + mu * closed, rtol=1e-13, atol=1e-13)
    M2, U2 = ref.momentum_update(np.ones((2, 2)), np.full((2, 2), 3.0), 0.5, nesterov=False)
    assert np.all(M2 == 3.5) and np.all(U2 == 3.5)


@pytest.mark.parametrize("rows,cols,scale", [(16, 4, 2.0), (4, 16, 1.0), (9, 9, 1.0), (36, 4, 3.0)])
def test_update_scale_and_direction(rows, cols, scale):
    # U with orthonormal short-side vectors: every normalised singular value is 1/sqrt(m)
    m = min(rows, cols)
    Q, _ = np.linalg.qr(np.random.default_rng(rows * 31 + cols).standard_normal((max(rows, cols), m)))
    U = Q if rows >= cols else Q.T
    W = np.random.default_rng(1).standard_normal((rows, cols))
    lr = 0.02
    W2, M2, X = ref.muon_step(W, U, np.zeros_like(U), lr=lr, mu=0.95, nesterov=False, ns_steps=5)
    fx = f_scalar(1.0 / (math.sqrt(m) + 1e-7), 5)
    np.testing.assert_allclose(X, fx * U, rtol=0, atol=1e-13)
    np.testing.assert_allclose(W2, W - lr * scale * fx * U, rtol=0, atol=1e-13)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
        np.array([0.0, -0.0, 1.0, -2.5, 3.0e38, -3.3e38, 1e-39, -1e-40, 1e-45]),
    ]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = ref.round_to_dtype(x.astype(np.float64), "bf16")
    np.testing.assert_array_equal(got, want)


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert ref.round_to_dtype(np.array([1 + 2 ** -8]), "bf16")[0] == 1.0
    # 1 + 3*2^-8 is halfway between 1+2^-7 and 1+2^-6: goes to 1+2^-6 (even)
    assert ref.round_to_dtype(np.array([1 + 3 * 2 ** -8]), "bf16")[0] == 1 + 2 ** -6
    # just above a tie rounds up
    assert ref.round_to_dtype(np.array([1 + 2 ** -8 + 2 ** -30]), "bf16")[0] == 1 + 2 ** -7


def test_golden_tiny_step_regression():
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_step.json")
    gold = json.load(open(path))
    h = gold["hyper"]
    for case in gold["cases"]:
        W, G, M = (np.array(case[k]) for k in ("W", "G", "M"))
        W2, M2, X = ref.muon_step(W, G, M, lr=h["lr"], mu=h["mu"], nesterov=h["nesterov"],
                                  ns_steps=h["ns_steps"], coeffs=tuple(h["coeffs"]), eps=h["eps"])
        np.testing.assert_allclose(W2, np.array(case["W_new"]), rtol=0, atol=1e-14)
        np.testing.assert_allclose(M2, np.array(case["M_new"]), rtol=0, atol=1e-14)
        np.testing.assert_allclose(X, np.array(case["X"]), rtol=0, atol=1e-14)
        # and the stored X is itself the scalar map of the normalised singular values
        np.testing.assert_allclose(np.array(case["X"]), spectral_expected(G + h["mu"] * (h["mu"] * M + G), h["ns_steps"]),
                                   rtol=0, atol=1e-11)


@pytest.mark.parametrize("shape", [(4, 9), (16, 40), (32, 112), (5, 5), (1, 8)])
def test_gram_space_recurrence_equals_the_iteration(shape):
    # X_S = Q_S X_0 with Q, G polynomials in X_0 X_0^T: the identity holds exactly in exact arithmetic
    for seed in range(5):
        U = np.random.default_rng(seed).standard_normal(shape)
        X0 = U / np.linalg.norm(U)
        steps = [ref.DEFAULT_COEFFS] * 5
        np.testing.assert_allclose(ref.newton_schulz_gram(X0, steps), ref.newton_schulz(X0, steps), rtol=0,
                                   atol=1e-11)
        # and against the scalar map of the singular values
        np.testing.assert_allclose(ref.newton_schulz_gram(X0, steps), spectral_expected(U, 5, eps=0.0), rtol=0,
                                   atol=1e-10)
