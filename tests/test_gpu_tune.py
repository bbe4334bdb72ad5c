"""Init-time tuning (DMUON_FLAG_TUNE): per-bucket tile widths chosen by
measurement, tile lists ordered by measured cost, results still match the
oracle, and the measured per-matrix costs drive the owner assignment."""

import numpy as np
import pytest
import torch

from matrix_optimizer_update_gb300 import dmuon as dm

from helpers import LibRun, TOL_M, TOL_X
from test_gpu_parity import _fill, compare

pytestmark = pytest.mark.gpu

SHAPES = [(1408, 2048)] * 6 + [(2048, 1408)] * 3 + [(512, 2048)] * 2 + [(640, 640)] * 2


@pytest.mark.parametrize("gram", [False, True])
def test_tuned_plan_matches_oracle_and_reports_costs(gram):
    run = LibRun(SHAPES, capture=True, gram_ns=gram)
    # rebind the same plan with tuning on
    muon = dm.Muon.create(SHAPES, flags=dm.FLAG_CAPTURE_UPDATE | dm.FLAG_TUNE | (dm.FLAG_GRAM_NS if gram else 0))
    run.muon = muon
    d = muon.plan.describe()
    assert d["tuned"] and d["tune_timed_buckets"] + d["tune_cached_buckets"] == len(d["buckets"])
    for b in d["buckets"]:
        assert b["bn_sym"] in (128, 256) and b["bn_gemm"] in (128, 256), b
        assert not b["pair"] or b["bn_sym"] == b["bn_gemm"] == 256, b
        assert all(t > 0 for t in b["tile_ms"]), b
    init = _fill(run, 3100)
    run.step()
    torch.cuda.synchronize()
    assert run.status() == 0
    for i, (W0, G, M0) in enumerate(init):
        e = compare(run, i, W0, G, M0, compute="bf16", param="bf16")
        assert e["x"] <= TOL_X["bf16"] and e["m"] <= TOL_M and e["w_violations"] == 0, (i, e)
    costs = muon.plan.costs()
    assert len(costs) == len(SHAPES) and all(c > 0 for c in costs)
    # same shape, same cost; the 1408x2048 matrices cost more than the 512x2048 ones
    assert costs[0] == costs[1] and costs[0] > costs[9]
    own, load = dm.dmuon_assign_owners(SHAPES, 4, costs=costs)
    assert sorted(set(own)) == [0, 1, 2, 3]
    np.testing.assert_allclose(sum(load), sum(costs), rtol=1e-12)


def test_second_tuned_plan_reuses_the_cached_timings():
    shapes = [(1536, 8960), (8960, 1536), (1536, 1536), (256, 1536)]
    first = dm.Muon.create(shapes, flags=dm.FLAG_TUNE)
    second = dm.Muon.create(shapes, flags=dm.FLAG_TUNE)
    a, b = first.plan.describe(), second.plan.describe()
    assert b["tuned"] and b["tune_timed_buckets"] == 0 and b["tune_cached_buckets"] == len(b["buckets"])
    # the same choices and per-tile costs as the plan that timed them
    key = ("m", "n", "pair", "bn_sym", "bn_gemm", "tile_ms")
    assert [{k: x[k] for k in key} for x in a["buckets"]] == [{k: x[k] for k in key} for x in b["buckets"]]
