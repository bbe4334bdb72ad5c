"""Binding a plan again: a bind that fails at any point leaves the plan
unbound (its steps are refused, never run on stale tables or on another
workspace), and a later successful bind gives the same results as a plan that
never failed. The failures are injected on the host (DMUON_TEST_FAIL) or come
from an argument the host check rejects; nothing faults on the GPU."""

import pytest
import torch

from matrix_optimizer_update_gb300 import dmuon as dm
from matrix_optimizer_update_gb300.inputs import random_matrix

from helpers import LibRun

pytestmark = pytest.mark.gpu

SHAPES = [(256, 384), (300, 700), (384, 256)]


def fill(run):
    for i, (r, c) in enumerate(SHAPES):
        run.set(i, W=random_matrix(r, c, 500 + i, 0.02, "cuda", "bf16"),
                G=random_matrix(r, c, 600 + i, 1e-3, "cuda", "bf16"))


def rebind(run, stream):
    nbytes = run.muon.plan.workspace_bytes()
    base = (run.muon.workspace.data_ptr() + 1023) // 1024 * 1024
    run.muon.plan.bind(base, nbytes, stream)


@pytest.mark.parametrize("point", ["bind_check", "bind_tables", "bind_maps", "bind_staging"])
def test_failed_rebind_unbinds_and_a_later_bind_recovers(point, monkeypatch):
    stream = torch.cuda.current_stream().cuda_stream
    ref_run, run = LibRun(SHAPES), LibRun(SHAPES)
    fill(ref_run)
    fill(run)
    ref_run.step()
    run.step()  # bound and stepped once
    monkeypatch.setenv("DMUON_TEST_FAIL", point)
    with pytest.raises(dm.DmuonError) as e:
        rebind(run, stream)
    assert e.value.status == dm.ERR_CUDA and point in str(e.value)
    monkeypatch.delenv("DMUON_TEST_FAIL")
    with pytest.raises(dm.DmuonError) as e:
        run.step()
    assert e.value.status == dm.ERR_NOT_BOUND
    rebind(run, stream)
    ref_run.step()
    run.step()
    torch.cuda.synchronize()
    assert run.status() == 0 and ref_run.status() == 0
    assert torch.equal(run.W, ref_run.W) and torch.equal(run.M, ref_run.M)
    for i in range(len(SHAPES)):
        assert torch.equal(run.update(i), ref_run.update(i))


def test_rebind_on_host_memory_unbinds():
    stream = torch.cuda.current_stream().cuda_stream
    run = LibRun(SHAPES)
    fill(run)
    run.step()
    nbytes = run.muon.plan.workspace_bytes()
    host = torch.empty(nbytes + 1024, dtype=torch.uint8, pin_memory=True)
    base = (host.data_ptr() + 1023) // 1024 * 1024
    with pytest.raises(dm.DmuonError) as e:
        run.muon.plan.bind(base, nbytes, stream)
    assert e.value.status == dm.ERR_WORKSPACE
    with pytest.raises(dm.DmuonError) as e:
        run.step()
    assert e.value.status == dm.ERR_NOT_BOUND
    rebind(run, stream)
    run.step()
    torch.cuda.synchronize()
    assert run.status() == 0
