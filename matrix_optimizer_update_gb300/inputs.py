"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and lays them out; it contains none of
the update's arithmetic. Both the CUDA path and the oracle receive the very
same bits: tensors are drawn once (on any torch device) and the oracle gets a
host copy.

Seeding: tensor t of matrix i in workload w uses
``seed = 1000 * w.index + 3 * i + t`` with t = 0 (gradient), 1 (weight),
2 (momentum history). Values: gradients N(0, grad_std), weights
N(0, weight_std) (second argument = standard deviation), drawn in fp32 and
rounded to the storage dtype. MoE expert gradients are multiplied by a
per-expert scale 10**U(log10 lo, log10 hi) from a seeded host generator
(numpy PCG64, seed 1000 * w.index + 999). Momentum is zero, or, for the
"history3" recipe, the fp32 sum mu^2*G1 + mu*G2 + G3 of three further seeded
gradient draws (the state three earlier steps would have left).

Every tensor of a kind lives in one flat buffer, with each matrix starting on a
256-element boundary (16-byte aligned for every dtype); ``views`` gives the
per-matrix ``rows x cols`` views.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from .workloads import Workload

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}
ALIGN_ELEMS = 256


def layout(shapes, align: int = ALIGN_ELEMS):
    """Element offsets of each matrix inside a flat buffer, and the total size."""
    offs, off = [], 0
    for r, c in shapes:
        offs.append(off)
        off += -(-(r * c) // align) * align
    return offs, off


@dataclass
class MatrixSet:
    shapes: list
    offsets: list
    W: torch.Tensor        # flat params (param dtype)
    G: torch.Tensor        # flat grads (grad dtype)
    M: torch.Tensor        # flat momentum (fp32)

    def view(self, flat: torch.Tensor, i: int) -> torch.Tensor:
        r, c = self.shapes[i]
        o = self.offsets[i]
        return flat[o:o + r * c].view(r, c)

    def views(self, flat: torch.Tensor):
        return [self.view(flat, i) for i in range(len(self.shapes))]

    def ptrs(self, flat: torch.Tensor):
        base = flat.data_ptr()
        es = flat.element_size()
        return [base + o * es for o in self.offsets]


def expert_scales(w: Workload) -> np.ndarray:
    """Per-(layer, expert) gradient scales, log-uniform in ``w.expert_scale``."""
    if not w.expert_scale:
        return np.ones((w.layers, max(w.experts, 1)))
    lo, hi = w.expert_scale
    rng = np.random.default_rng(1000 * w.index + 999)
    u = rng.uniform(np.log10(lo), np.log10(hi), size=(w.layers, w.experts))
    return 10.0 ** u


def _normal(shape, std, seed, device, out_dtype, draws: int = 1):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    outs = []
    for _ in range(draws):
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        outs.append(t if out_dtype == torch.float32 else t.to(out_dtype))
    return outs


def make_matrix_set(w: Workload, device="cuda", seed_offset: int = 0,
                    only=None) -> MatrixSet:
    """Draw the workload's W, G and M on ``device``.

    ``seed_offset`` shifts every seed (used to give each replica its own
    data). ``only`` (a set of matrix indices) draws just those matrices and
    leaves the others zero: for quick tests that sample a few matrices.
    """
    mats = list(w.matrices())
    shapes = [(r, c) for _, _, r, c, _ in mats]
    offs, total = layout(shapes)
    pdt, gdt = TORCH_DTYPE[w.param_dtype], TORCH_DTYPE[w.grad_dtype]
    W = torch.zeros(total, dtype=pdt, device=device)
    G = torch.zeros(total, dtype=gdt, device=device)
    M = torch.zeros(total, dtype=torch.float32, device=device)
    ms = MatrixSet(shapes, offs, W, G, M)
    scales = expert_scales(w)
    base = 1000 * w.index + seed_offset
    for i, (layer, role, r, c, e) in enumerate(mats):
        if only is not None and i not in only:
            continue
        std = w.grad_std if e < 0 else float(scales[layer, e])
        (g,) = _normal((r, c), std, base + 3 * i + 0, device, gdt)
        ms.view(G, i).copy_(g)
        (wt,) = _normal((r, c), w.weight_std, base + 3 * i + 1, device, pdt)
        ms.view(W, i).copy_(wt)
        if w.momentum_init == "history3":
            g1, g2, g3 = _normal((r, c), std, base + 3 * i + 2, device, gdt, draws=3)
            mu = w.mu
            hist = (mu * mu) * g1.float() + mu * g2.float() + g3.float()
            ms.view(M, i).copy_(hist)
    return ms


def random_matrix(rows, cols, seed, std=1.0, device="cpu", dtype="f32"):
    """One seeded N(0, std) matrix (for small tests)."""
    (t,) = _normal((rows, cols), std, seed, device, TORCH_DTYPE[dtype])
    return t
