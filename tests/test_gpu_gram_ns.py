"""GPU parity of the Gram-space form of the iteration (DMUON_FLAG_GRAM_NS)
against the fp64 oracle: wide matrices iterate on G = X X^T and meet the same
tolerances as the standard form; square matrices keep the standard form."""

import pytest
import torch

from helpers import LibRun
from test_gpu_parity import RAGGED, _check_all, _fill

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("compute", ["bf16", "f32"])
def test_gram_form_ragged_shapes(compute):
    prm = "bf16" if compute == "bf16" else "f32"
    run = LibRun(RAGGED, param=prm, grad=prm, compute=compute, gram_ns=True)
    forms = {(b["m"], b["n"]): b["form"] for b in run.muon.plan.describe()["buckets"]}
    assert forms[(130, 130)] == "standard" and forms[(300, 700)] == "gram" and forms[(129, 257)] == "standard"
    init = _fill(run, 700, grad_std=1e-3 if compute == "bf16" else 1.0, w_std=0.02 if compute == "bf16" else 1.0,
                 m_std=1e-3)
    run.step()
    torch.cuda.synchronize()
    worst = _check_all(run, init)
    assert run.status() == 0
    print("gram", compute, worst)


@pytest.mark.parametrize("ns_steps", [1, 2, 3, 5])
@pytest.mark.parametrize("compute", ["bf16", "f32"])
def test_gram_form_step_counts(ns_steps, compute):
    shapes = [(200, 600), (600, 200), (64, 64), (128, 1000)]
    prm = "bf16" if compute == "bf16" else "f32"
    run = LibRun(shapes, param=prm, grad=prm, compute=compute, ns_steps=ns_steps, gram_ns=True)
    init = _fill(run, 1900 + ns_steps)
    run.step()
    torch.cuda.synchronize()
    _check_all(run, init, ns_steps=ns_steps)


def test_gram_form_per_step_coeffs():
    coeffs = [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.0, -1.5, 0.5)]
    shapes = [(256, 768), (768, 256)]
    for compute in ("bf16", "f32"):
        run = LibRun(shapes, param="f32", grad="f32", compute=compute, ns_steps=3, coeffs=coeffs, gram_ns=True)
        init = _fill(run, 2300, m_std=1e-3)
        run.step()
        torch.cuda.synchronize()
        _check_all(run, init, ns_steps=3, coeffs=coeffs)
