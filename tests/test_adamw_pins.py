"""Pins of the AdamW oracle: torch.optim.AdamW in float64 (a library
routine), and closed forms of the first step and of a constant gradient."""

import numpy as np
import pytest
import torch

from oracle.adamw_ref import adamw_step


@pytest.mark.parametrize("wd", [0.0, 0.01, 0.1])
def test_matches_torch_adamw_float64(wd):
    rng = np.random.default_rng(0)
    p0 = rng.standard_normal(1000)
    grads = [rng.standard_normal(1000) * 10.0 ** rng.uniform(-4, 0) for _ in range(7)]
    t = torch.tensor(p0.copy(), dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([t], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=wd, foreach=False)
    p, m, v = p0.copy(), np.zeros(1000), np.zeros(1000)
    for k, g in enumerate(grads, start=1):
        t.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = adamw_step(p, g, m, v, lr=1e-3, weight_decay=wd, step=k)
        np.testing.assert_allclose(p, t.detach().numpy(), rtol=1e-13, atol=1e-15)
        st = opt.state[t]
        np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-12, atol=1e-17)  # torch blends with lerp
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-12, atol=1e-17)


def test_first_step_closed_form():
    # zero state, t = 1: the bias-corrected moments are g and g^2, so the step is lr * g / (|g| + eps)
    g = np.array([1e-3, -2.0, 0.0, 5e-9, -7.5])
    p0 = np.array([0.5, -0.25, 1.0, 2.0, 0.0])
    p, m, v = adamw_step(p0, g, np.zeros(5), np.zeros(5), lr=0.01, weight_decay=0.1, step=1)
    want = p0 * (1 - 0.01 * 0.1) - 0.01 * g / (np.abs(g) + 1e-8)
    np.testing.assert_allclose(p, want, rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(m, 0.1 * g, rtol=1e-15)
    np.testing.assert_allclose(v, 0.001 * g * g, rtol=1e-13)


def test_constant_gradient_closed_form():
    # with a constant g the bias-corrected moments stay exactly g and g^2 at every step
    g = np.array([0.3, -1e-4, 2.0])
    p, m, v = np.zeros(3), np.zeros(3), np.zeros(3)
    lr = 1e-2
    for k in range(1, 30):
        p, m, v = adamw_step(p, g, m, v, lr=lr, weight_decay=0.0, step=k)
        np.testing.assert_allclose(m / (1 - 0.9 ** k), g, rtol=1e-12)
        np.testing.assert_allclose(v / (1 - 0.999 ** k), g * g, rtol=1e-10)
    np.testing.assert_allclose(p, -29 * lr * g / (np.abs(g) + 1e-8), rtol=1e-9)
