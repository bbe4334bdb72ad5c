"""Synthetic matrix sets the library is tested and measured on.

Each workload is the list of 2-D projection matrices of a model (stored
``rows x cols``, rows = dim 0) repeated over its layers, with the dtypes and
value distributions of the inputs. The models are the ones the DMuon pages
train (project docs, "what DMuon can do": Qwen2.5 1.5B-7B and Llama-3 3B-8B on
8xA800; MoE: one owner per expert projection). No weights or datasets are
used: every tensor is drawn from a seeded generator (see ``inputs.py``).

This module holds shapes and bookkeeping only (counts, flop and byte totals
for reporting); none of the update's arithmetic lives here.
"""

from __future__ import annotations

from dataclasses import dataclass, field

QUINTIC = (3.4445, -4.7750, 2.0315)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                      # seed namespace (1-based)
    layer_shapes: tuple             # ((role, rows, cols), ...) for one layer
    layers: int
    param_dtype: str                # "f32" | "bf16"
    grad_dtype: str                 # "f32" | "bf16"
    compute: str                    # "f32" (fp32 math) | "bf16" (bf16 operands, fp32 accumulate)
    grad_std: float
    weight_std: float
    momentum_init: str = "zero"     # "zero" | "history3"
    expert_scale: tuple | None = None   # (lo, hi) log-uniform per-expert grad scale
    experts: int = 0                # experts per layer (MoE); expert roles are tagged "e:"
    lr: float = 0.02
    mu: float = 0.95
    nesterov: bool = True
    ns_steps: int = 5
    coeffs: tuple = QUINTIC
    eps: float = 1e-7
    description: str = ""

    def matrices(self):
        """Yield ``(layer, role, rows, cols, expert)`` for every matrix, in order."""
        for layer in range(self.layers):
            for role, r, c in self.layer_shapes:
                if role.startswith("e:"):
                    for e in range(self.experts):
                        yield layer, role[2:], r, c, e
                else:
                    yield layer, role, r, c, -1

    @property
    def shapes(self):
        return [(r, c) for _, _, r, c, _ in self.matrices()]

    @property
    def per_layer(self) -> int:
        n = 0
        for role, _, _ in self.layer_shapes:
            n += self.experts if role.startswith("e:") else 1
        return n


WORKLOADS = {
    "toy": Workload(
        name="toy", index=1,
        layer_shapes=(("w", 128, 256),), layers=4,
        param_dtype="f32", grad_dtype="f32", compute="f32",
        grad_std=1.0, weight_std=1.0,
        description="4 fp32 matrices 128x256, N(0,1) grads and weights, zero momentum, fp32 math",
    ),
    "qwen2.5-1.5b": Workload(
        name="qwen2.5-1.5b", index=2,
        layer_shapes=(("q", 1536, 1536), ("k", 256, 1536), ("v", 256, 1536), ("o", 1536, 1536),
                      ("gate", 8960, 1536), ("up", 8960, 1536), ("down", 1536, 8960)),
        layers=28, param_dtype="bf16", grad_dtype="bf16", compute="bf16",
        grad_std=1e-3, weight_std=0.02,
        description="Qwen2.5-1.5B projection set, 28 layers, 196 matrices",
    ),
    "llama-3.2-3b": Workload(
        name="llama-3.2-3b", index=3,
        layer_shapes=(("q", 3072, 3072), ("k", 1024, 3072), ("v", 1024, 3072), ("o", 3072, 3072),
                      ("gate", 8192, 3072), ("up", 8192, 3072), ("down", 3072, 8192)),
        layers=28, param_dtype="bf16", grad_dtype="bf16", compute="bf16",
        grad_std=1e-3, weight_std=0.02, momentum_init="history3",
        description="Llama-3.2-3B projection set, 28 layers, 196 matrices, momentum from 3 prior seeded grads",
    ),
    "llama-3.1-8b": Workload(
        name="llama-3.1-8b", index=4,
        layer_shapes=(("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
                      ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)),
        layers=32, param_dtype="bf16", grad_dtype="bf16", compute="bf16",
        grad_std=1e-3, weight_std=0.02,
        description="Llama-3.1-8B projection set, 32 layers, 224 matrices",
    ),
    "moe-16x64": Workload(
        name="moe-16x64", index=5,
        layer_shapes=(("q", 2048, 2048), ("k", 512, 2048), ("v", 512, 2048), ("o", 2048, 2048),
                      ("e:gate", 1408, 2048), ("e:up", 1408, 2048), ("e:down", 2048, 1408)),
        layers=16, experts=64, param_dtype="bf16", grad_dtype="bf16", compute="bf16",
        grad_std=1e-3, weight_std=0.02, expert_scale=(1e-5, 1e-2),
        description="MoE ragged set: 16 layers x 64 experts x (gate, up, down) + attention, 3136 matrices",
    ),
}


def get(name: str) -> Workload:
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; choose from {sorted(WORKLOADS)}") from None


# --------------------------------------------------------------------------
# reporting arithmetic (work counts, not the update itself)
# --------------------------------------------------------------------------

def ns_flops(rows: int, cols: int, ns_steps: int) -> int:
    """Algorithmic Newton-Schulz flops of one matrix, counting the symmetric
    products once (only one triangle of X X^T and of A A^T is computed):
    ``S * [m(m+1)n + m^2(m+1) + 2 m^2 n]`` with m = min, n = max."""
    m, n = min(rows, cols), max(rows, cols)
    return ns_steps * (m * (m + 1) * n + m * m * (m + 1) + 2 * m * m * n)


def ns_flops_dense(rows: int, cols: int, ns_steps: int) -> int:
    """Dense-equivalent flops ``S * (4 m^2 n + 2 m^3)`` (printed for context only)."""
    m, n = min(rows, cols), max(rows, cols)
    return ns_steps * (4 * m * m * n + 2 * m ** 3)


def phase_flops(rows: int, cols: int) -> dict:
    """Per Newton-Schulz step, algorithmic flops of the three products."""
    m, n = min(rows, cols), max(rows, cols)
    return {"gram": m * (m + 1) * n, "poly": m * m * (m + 1), "gemm": 2 * m * m * n}


def stream_bytes(rows: int, cols: int, grad_bytes: int, param_bytes: int, x_bytes: int) -> dict:
    """Algorithmic HBM bytes of the streaming work of one matrix: the momentum
    pass reads G and M, writes M and the normalised-orientation copy U; the
    update reads and writes W."""
    e = rows * cols
    return {"momentum": e * (grad_bytes + 4 + 4 + x_bytes), "update": e * 2 * param_bytes}


DTYPE_BYTES = {"f32": 4, "bf16": 2}


def totals(w: Workload) -> dict:
    shapes = w.shapes
    return {
        "matrices": len(shapes),
        "params": sum(r * c for r, c in shapes),
        "ns_flops": sum(ns_flops(r, c, w.ns_steps) for r, c in shapes),
        "ns_flops_dense": sum(ns_flops_dense(r, c, w.ns_steps) for r, c in shapes),
    }
