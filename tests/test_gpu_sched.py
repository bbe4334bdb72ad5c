"""Tile scheduling of the tensor-core launches.

By default each CTA (each CTA pair of the two-SM kernel) claims its next tile
from the launch's counter when it becomes free (tiles in cost order, largest
first); DMUON_FLAG_STATIC_TILES deals the same list round-robin instead. Which
CTA computes a tile does not change how the tile is computed, so both
schedules must give the same bits. The per-CTA timing records must cover
every CTA of a launch."""

import pytest
import torch

from matrix_optimizer_update_gb300 import dmuon as dm
from matrix_optimizer_update_gb300.inputs import random_matrix

from helpers import LibRun

pytestmark = pytest.mark.gpu

SHAPES = [(1408, 2048), (2048, 1408), (512, 2048), (300, 700), (700, 300), (129, 257), (1024, 1024), (64, 64)]


def fill(run, seed):
    for i, (r, c) in enumerate(run.shapes):
        run.set(i, W=random_matrix(r, c, seed + 3 * i, 0.02, "cuda", run.param),
                G=random_matrix(r, c, seed + 3 * i + 1, 1e-3, "cuda", run.grad),
                M=random_matrix(r, c, seed + 3 * i + 2, 1e-3, "cuda", "f32"))


@pytest.mark.parametrize("form", ["standard", "gram", "aX"])
def test_claimed_and_dealt_tiles_agree_bitwise(form):
    kw = {"gram_ns": form == "gram", "epilogue_ax": form == "aX"}
    a = LibRun(SHAPES, **kw)
    b = LibRun(SHAPES, flags=dm.FLAG_STATIC_TILES, **kw)
    fill(a, 7700)
    b.W.copy_(a.W)
    b.G.copy_(a.G)
    b.M.copy_(a.M)
    for _ in range(3):  # the counters reset themselves launch after launch
        a.step()
        b.step()
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(a.W, b.W) and torch.equal(a.M, b.M)
    for i in range(len(SHAPES)):
        assert torch.equal(a.update(i), b.update(i)), i


@pytest.mark.parametrize("form", ["standard", "gram"])
def test_claimed_and_dealt_pair_tiles_agree_bitwise(form, monkeypatch):
    """The two-SM kernel: the leader of each pair claims, and hands every item to its peer."""
    monkeypatch.setenv("DMUON_TEST_FORCE_PAIRS", "1")  # pairs on every bucket with a short side >= 256
    a = LibRun(SHAPES, pair=True, gram_ns=form == "gram")
    b = LibRun(SHAPES, pair=True, gram_ns=form == "gram", flags=dm.FLAG_STATIC_TILES)
    monkeypatch.delenv("DMUON_TEST_FORCE_PAIRS")
    assert sum(B["pair"] for B in a.muon.plan.describe()["buckets"]) >= 4
    fill(a, 7900)
    b.W.copy_(a.W)
    b.G.copy_(a.G)
    b.M.copy_(a.M)
    for _ in range(3):
        a.step()
        b.step()
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(a.W, b.W) and torch.equal(a.M, b.M)
    for i in range(len(SHAPES)):
        assert torch.equal(a.update(i), b.update(i)), i


@pytest.mark.parametrize("pair", [False, True])
def test_cta_times_cover_every_cta(pair, monkeypatch):
    if pair:
        monkeypatch.setenv("DMUON_TEST_FORCE_PAIRS", "1")
    run = LibRun(SHAPES, capture=False, pair=pair)
    monkeypatch.delenv("DMUON_TEST_FORCE_PAIRS", raising=False)
    fill(run, 7800)
    plan = run.muon.plan
    launches = plan.describe()["launches"]
    plan.profile_cta_times(True)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    run.step()
    t1.record()
    torch.cuda.synchronize()
    step_ms = t0.elapsed_time(t1)
    stream = torch.cuda.current_stream().cuda_stream
    seen = 0
    for li, L in enumerate(launches):
        rec = plan.read_cta_times(li, stream)
        if L["kind"] in (dm.KIND_MOMENTUM, dm.KIND_NORM):
            assert rec == []
            continue
        assert len(rec) == (2 if L["pair"] else 1) * L["grid"], (li, len(rec), L["grid"])
        for start, end in rec:
            assert 0 < start <= end and (end - start) * 1e-6 <= step_ms + 1.0, (li, start, end)
        seen += 1
    assert seen == len(launches) - 2
    plan.profile_cta_times(False)
    assert run.status() == 0
