"""Poison-filled workspace: every element a step reads must have been written
earlier in the same step (or, for the tables, by bind).

The whole workspace is filled with 0xFF bytes (NaN in bf16 and in fp32)
before bind, and the step's scratch regions (per-matrix s, partial sums, every
bucket buffer, the update capture) are filled again between two steps. A tile
that a phase never writes, a mirrored lower-triangle element that is missed,
or a read past what the step produced then shows up as NaN in the results. The
results must match the fp64 oracle as on a clean workspace, with no device
status bit set."""

import numpy as np
import pytest
import torch

from matrix_optimizer_update_gb300 import dmuon as dm
from matrix_optimizer_update_gb300 import workloads as wl
from matrix_optimizer_update_gb300.inputs import TORCH_DTYPE, layout, make_matrix_set, random_matrix
from oracle import muon_ref as ref

from helpers import TOL_M, rel, tol_x, weight_rounding_violations

pytestmark = pytest.mark.gpu

POISON = 0xFF


class PoisonRun:
    """A plan bound to a workspace that was filled with NaN bytes before bind."""

    def __init__(self, shapes, *, param="bf16", grad="bf16", compute="bf16", flags=0, ns_steps=5):
        self.shapes = list(shapes)
        self.param, self.compute, self.ns_steps = param, compute, ns_steps
        self.plan = dm.dmuon_plan(self.shapes, ns_steps, param=param, grad=grad, compute=compute,
                                  flags=flags | dm.FLAG_CAPTURE_UPDATE)
        nbytes = self.plan.workspace_bytes()
        self.ws = torch.full((nbytes + 1024,), POISON, dtype=torch.uint8, device="cuda")
        self.base = (self.ws.data_ptr() + 1023) // 1024 * 1024
        self.off0 = self.base - self.ws.data_ptr()
        self.plan.bind(self.base, nbytes, torch.cuda.current_stream().cuda_stream)
        self.regions = self.plan.describe()["regions"]
        self.offs, total = layout(self.shapes)
        self.W = torch.zeros(total, dtype=TORCH_DTYPE[param], device="cuda")
        self.G = torch.zeros(total, dtype=TORCH_DTYPE[grad], device="cuda")
        self.M = torch.zeros(total, dtype=torch.float32, device="cuda")

    def poison_scratch(self):
        for off, n in self.regions["scratch"]:
            self.ws[self.off0 + off:self.off0 + off + n].fill_(POISON)

    def view(self, flat, i):
        r, c = self.shapes[i]
        return flat[self.offs[i]:self.offs[i] + r * c].view(r, c)

    def ptrs(self, flat):
        return [flat.data_ptr() + o * flat.element_size() for o in self.offs]

    def step(self):
        s = torch.cuda.current_stream().cuda_stream
        self.plan.step(self.ptrs(self.W), self.ptrs(self.G), self.ptrs(self.M), 0.02, 0.95, True, s)

    def update(self, i):
        r, c = self.shapes[i]
        out = torch.empty(r, c, dtype=torch.float32, device="cuda")
        self.plan.read_update(i, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        return out.double().cpu().numpy()


def check_two_steps(run, idx=None):
    """Two steps, the scratch poisoned again in between; oracle parity after each."""
    idx = range(len(run.shapes)) if idx is None else idx
    host = {i: [run.view(run.W, i).double().cpu().numpy(), run.view(run.M, i).double().cpu().numpy()] for i in idx}
    for step in range(2):
        if step:
            run.poison_scratch()
        G = {i: run.view(run.G, i).double().cpu().numpy() for i in idx}
        run.step()
        torch.cuda.synchronize()
        assert run.plan.read_device_status(torch.cuda.current_stream().cuda_stream) == 0
        for i in idx:
            r, c = run.shapes[i]
            W0, M0 = host[i]
            Wr, Mr, Xr = ref.muon_step(W0, G[i], M0, lr=0.02, mu=0.95, nesterov=True, ns_steps=run.ns_steps)
            Xg = run.update(i)
            Wg = run.view(run.W, i).double().cpu().numpy()
            Mg = run.view(run.M, i).double().cpu().numpy()
            assert np.isfinite(Xg).all() and np.isfinite(Wg).all(), (step, i)
            assert rel(Xg, Xr) <= tol_x(run.compute, min(r, c)), (step, i, rel(Xg, Xr))
            assert rel(Mg, Mr) <= TOL_M, (step, i)
            assert weight_rounding_violations(Wg, Wr, W0, Xg, Xr, 0.02 * ref.update_scale(r, c), run.param) == 0
            host[i] = [Wg, Mg]


RAGGED = [(300, 700), (700, 300), (129, 257), (256, 384), (384, 256), (1408, 2048), (2048, 1408), (520, 1000),
          (64, 64), (8, 24)]


def fill(run, seed):
    for i, (r, c) in enumerate(run.shapes):
        run.view(run.W, i).copy_(random_matrix(r, c, seed + 2 * i, 0.02, "cuda", run.param))
        run.view(run.G, i).copy_(random_matrix(r, c, seed + 2 * i + 1, 1e-3, "cuda", run.param))


@pytest.mark.parametrize("form", ["one_sm", "gram", "pair", "aX", "fp32"])
def test_poisoned_workspace_ragged_shapes(form):
    flags = {"one_sm": dm.FLAG_ONE_SM_TILES, "gram": dm.FLAG_GRAM_NS, "pair": 0, "aX": dm.FLAG_EPILOGUE_AX,
             "fp32": 0}[form]
    dt = "f32" if form == "fp32" else "bf16"
    shapes = RAGGED + ([(512, 1024), (1024, 512), (768, 2048)] if form == "pair" else [])
    run = PoisonRun(shapes, param=dt, grad=dt, compute=dt, flags=flags)
    fill(run, 9100)
    check_two_steps(run)


@pytest.mark.parametrize("ns_steps", [0, 1, 2])
def test_poisoned_workspace_short_iterations(ns_steps):
    run = PoisonRun(RAGGED[:6], ns_steps=ns_steps)
    fill(run, 9200)
    check_two_steps(run)


def test_poisoned_workspace_moe_full_size():
    """One full-size MoE matrix set (3136 matrices) on a poisoned workspace, sampled against the oracle."""
    w = wl.get("moe-16x64")
    run = PoisonRun(w.shapes)
    ms = make_matrix_set(w, "cuda")
    run.W.copy_(ms.W)
    run.G.copy_(ms.G)
    run.M.copy_(ms.M)
    del ms
    mats = list(w.matrices())
    idx = [i for i, m in enumerate(mats) if m[0] == 0 and (m[4] < 0 or m[4] in (0, 63))]
    idx += [i for i, m in enumerate(mats) if m[0] == w.layers - 1 and m[4] in (-1, 31)]
    check_two_steps(run, idx)
    assert bool(torch.isfinite(run.W).all())  # every matrix, not only the sampled ones
