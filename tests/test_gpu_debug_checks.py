"""Host-side debug checks (DMUON_FLAG_DEBUG_CHECKS): after every launch the
library recomputes sampled output elements on the host. On correct kernels
they must never fire, and the results must be the same bits as without the
checks; with one launch left out (a host-side test hook, on a workspace
poisoned with NaN bytes), the check after it must report the stale output."""

import pytest
import torch

from matrix_optimizer_update_gb300 import dmuon as dm
from matrix_optimizer_update_gb300.inputs import random_matrix

from helpers import LibRun

pytestmark = pytest.mark.gpu

SHAPES = [(300, 700), (700, 300), (129, 257), (1408, 2048), (256, 384), (64, 64)]


def fill(run, seed):
    for i, (r, c) in enumerate(run.shapes):
        run.set(i, W=random_matrix(r, c, seed + 3 * i, 0.02, "cuda", run.param),
                G=random_matrix(r, c, seed + 3 * i + 1, 1e-3, "cuda", run.grad),
                M=random_matrix(r, c, seed + 3 * i + 2, 1e-3, "cuda", "f32"))


@pytest.mark.parametrize("form", ["standard", "gram", "pair", "aX", "fp32", "ns0"])
def test_debug_checks_pass_and_change_nothing(form):
    dt = "f32" if form == "fp32" else "bf16"
    shapes = SHAPES + ([(512, 1024)] if form == "pair" else [])
    kw = dict(param=dt, grad=dt, compute=dt, gram_ns=form == "gram", pair=form == "pair", epilogue_ax=form == "aX",
              ns_steps=0 if form == "ns0" else 5)
    a = LibRun(shapes, flags=dm.FLAG_DEBUG_CHECKS, **kw)
    b = LibRun(shapes, **kw)
    fill(a, 8800)
    b.W.copy_(a.W)
    b.G.copy_(a.G)
    b.M.copy_(a.M)
    for _ in range(2):
        a.step()  # raises DmuonError if a check fails
        b.step()
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(a.W, b.W) and torch.equal(a.M, b.M)


@pytest.mark.parametrize("skip_kind", [dm.KIND_GRAM, dm.KIND_POLY, dm.KIND_GEMM])
def test_debug_checks_report_a_launch_left_out(skip_kind, monkeypatch):
    shapes = [(512, 1024), (1024, 512)]
    plan = dm.dmuon_plan(shapes, 5, flags=dm.FLAG_DEBUG_CHECKS)
    launches = plan.describe()["launches"]
    li = next(i for i, L in enumerate(launches) if L["kind"] == skip_kind)
    nbytes = plan.workspace_bytes()
    ws = torch.full((nbytes + 1024,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN in bf16
    base = (ws.data_ptr() + 1023) // 1024 * 1024
    stream = torch.cuda.current_stream().cuda_stream
    plan.bind(base, nbytes, stream)
    W = [random_matrix(r, c, 8900 + i, 0.02, "cuda", "bf16") for i, (r, c) in enumerate(shapes)]
    G = [random_matrix(r, c, 8950 + i, 1e-3, "cuda", "bf16") for i, (r, c) in enumerate(shapes)]
    M = [torch.zeros(r, c, device="cuda") for r, c in shapes]
    ptrs = lambda ts: [t.data_ptr() for t in ts]  # noqa: E731
    monkeypatch.setenv("DMUON_TEST_SKIP_LAUNCH", str(li))
    with pytest.raises(dm.DmuonError) as e:
        plan.step(ptrs(W), ptrs(G), ptrs(M), 0.02, 0.95, True, stream)
    assert e.value.status == dm.ERR_DEVICE and f"launch {li} " in str(e.value), str(e.value)
    monkeypatch.delenv("DMUON_TEST_SKIP_LAUNCH")
    torch.cuda.synchronize()
