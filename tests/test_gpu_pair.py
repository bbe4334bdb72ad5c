"""GPU parity of the two-SM tile path (DMUON_FLAG_PAIR_TILES: 256 x 256 tiles
on clusters of two CTAs, tcgen05 cta_group::2) against the fp64 oracle, in
both iteration forms, plus bitwise agreement of repeated runs."""

import pytest
import torch

from helpers import LibRun
from test_gpu_parity import _check_all, _fill

pytestmark = pytest.mark.gpu

# pair buckets: short side a multiple of 256 (512 x 1000 and 1000 x 512 with ragged long sides);
# the others run on one-SM tiles beside them
SHAPES = [(300, 700), (700, 300), (520, 1000), (256, 1536), (1536, 256), (512, 512), (384, 384), (130, 130),
          (512, 1000), (1000, 512)]


def test_pair_tiles_small():
    run = LibRun([(256, 512), (512, 256)], pair=True)
    d = run.muon.plan.describe()
    assert all(b["pair"] for b in d["buckets"])
    init = _fill(run, 5000)
    run.step()
    torch.cuda.synchronize()
    assert run.status() == 0
    _check_all(run, init)


@pytest.mark.parametrize("gram", [False, True])
def test_pair_tiles_ragged(gram):
    run = LibRun(SHAPES, pair=True, gram_ns=gram)
    pairs = {(b["m"], b["n"]): b["pair"] for b in run.muon.plan.describe()["buckets"]}
    assert pairs[(512, 512)] and pairs[(256, 1536)] and pairs[(512, 1000)]
    assert not pairs[(300, 700)] and not pairs[(130, 130)] and not pairs[(520, 1000)] and not pairs[(384, 384)]
    init = _fill(run, 5100, m_std=1e-3)
    run.step()
    torch.cuda.synchronize()
    assert run.status() == 0
    worst = _check_all(run, init)
    print("pair", "gram" if gram else "standard", worst)


@pytest.mark.parametrize("ns_steps", [1, 2])
def test_pair_tiles_step_counts(ns_steps):
    run = LibRun([(256, 768), (768, 256), (512, 512)], pair=True, ns_steps=ns_steps)
    init = _fill(run, 5200 + ns_steps)
    run.step()
    torch.cuda.synchronize()
    _check_all(run, init, ns_steps=ns_steps)


def test_pair_tiles_deterministic():
    run = LibRun([(512, 1024), (1024, 512)], pair=True, capture=False)
    _fill(run, 5300)
    W0, M0 = run.W.clone(), run.M.clone()
    run.step()
    W1, M1 = run.W.clone(), run.M.clone()
    run.W.copy_(W0)
    run.M.copy_(M0)
    run.step()
    assert torch.equal(run.W, W1) and torch.equal(run.M, M1)


def test_pair_tiles_with_ax_epilogue():
    """Pair tiles with the literal form of the step (a*X read in the last product's epilogue)."""
    run = LibRun([(512, 1000), (1000, 512), (256, 768)], pair=True, epilogue_ax=True)
    assert all(b["pair"] for b in run.muon.plan.describe()["buckets"])
    init = _fill(run, 5400, m_std=1e-3)
    run.step()
    torch.cuda.synchronize()
    assert run.status() == 0
    _check_all(run, init)


@pytest.mark.parametrize("param,grad", [("f32", "bf16"), ("bf16", "f32")])
def test_pair_tiles_mixed_storage(param, grad):
    """Pair tiles with fp32 weights (the per-row weight update) or fp32 gradients."""
    run = LibRun([(256, 512), (512, 256), (512, 1000)], param=param, grad=grad, compute="bf16", pair=True)
    init = _fill(run, 5500, m_std=1e-3)
    run.step()
    torch.cuda.synchronize()
    assert run.status() == 0
    _check_all(run, init)


@pytest.mark.parametrize("gram", [False, True])
def test_pair_and_one_sm_tiles_agree_bitwise(gram):
    """Two-SM and one-SM tiles sum every output element over K in the same order: the stored weights
    and momenta of both plans are identical, bit for bit."""
    shapes = [(512, 1024), (1024, 512), (256, 768)]
    a = LibRun(shapes, pair=False, gram_ns=gram, capture=False)
    b = LibRun(shapes, pair=True, gram_ns=gram, capture=False)
    assert all(x["pair"] for x in b.muon.plan.describe()["buckets"])
    _fill(a, 5600, m_std=1e-3)
    b.W.copy_(a.W)
    b.G.copy_(a.G)
    b.M.copy_(a.M)
    a.step()
    b.step()
    torch.cuda.synchronize()
    assert torch.equal(a.W, b.W) and torch.equal(a.M, b.M)


RAGGED_PAIRS = [(300, 700), (700, 300), (520, 1000), (1408, 2048), (2048, 1408), (640, 640), (384, 384)]


@pytest.mark.parametrize("gram", [False, True])
def test_pair_tiles_on_short_sides_not_a_multiple_of_256(gram, monkeypatch):
    """Pairs on short sides that leave the last row pair half empty (the second CTA's rows all past the
    matrix): what tuning may choose. Oracle parity, and the same bits as one-SM tiles."""
    monkeypatch.setenv("DMUON_TEST_FORCE_PAIRS", "1")
    run = LibRun(RAGGED_PAIRS, pair=True, gram_ns=gram)
    monkeypatch.delenv("DMUON_TEST_FORCE_PAIRS")
    assert all(b["pair"] for b in run.muon.plan.describe()["buckets"])
    one = LibRun(RAGGED_PAIRS, pair=False, gram_ns=gram)
    init = _fill(run, 5700, m_std=1e-3)
    one.W.copy_(run.W)
    one.G.copy_(run.G)
    one.M.copy_(run.M)
    run.step()
    one.step()
    torch.cuda.synchronize()
    assert run.status() == 0 and one.status() == 0
    _check_all(run, init)
    assert torch.equal(run.W, one.W) and torch.equal(run.M, one.M)
