"""GPU parity: the library (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element, at sizes the oracle finishes in
seconds that still span several tiles and ragged edges."""

import json
import os

import numpy as np
import pytest
import torch

from matrix_optimizer_update_gb300 import dmuon as dm
from matrix_optimizer_update_gb300 import workloads
from matrix_optimizer_update_gb300.inputs import make_matrix_set, random_matrix
from oracle import muon_ref as ref

from helpers import TOL_M, TOL_W, TOL_X, LibRun, compare, tol_x, weight_rounding_violations

pytestmark = pytest.mark.gpu

RAGGED = [(300, 700), (700, 300), (129, 257), (257, 129), (130, 130), (1, 37), (37, 1), (520, 1000),
          (8, 16), (16, 8), (256, 1536), (1536, 256), (3, 5)]


def _fill(run, seed, grad_std=1e-3, w_std=0.02, m_std=0.0):
    init = []
    for i, (r, c) in enumerate(run.shapes):
        G = random_matrix(r, c, seed + 3 * i, grad_std, "cuda", run.grad)
        W = random_matrix(r, c, seed + 3 * i + 1, w_std, "cuda", run.param)
        M = random_matrix(r, c, seed + 3 * i + 2, m_std, "cuda", "f32") if m_std else torch.zeros(r, c, device="cuda")
        run.set(i, W=W, G=G, M=M)
        init.append((W.double().cpu().numpy(), G.double().cpu().numpy(), M.double().cpu().numpy()))
    return init


def _check_all(run, init, **kw):
    """X within the mode's bound, momentum within 1e-6, and every stored weight
    equal to the exact update rounded once to its storage type (up to the
    update's own error). The 1e-3 relative-Frobenius bar on bf16 weights is
    asserted on the workload shapes (test_gpu_workloads.py): on small ad-hoc
    shapes the bf16 rounding of W alone puts that figure above 1e-3."""
    worst = {}
    for i, (W0, G, M0) in enumerate(init):
        e = compare(run, i, W0, G, M0, compute=run.compute, param=run.param, **kw)
        for k, v in e.items():
            worst[k] = max(worst.get(k, 0.0), v)
        assert e["x"] <= tol_x(run.compute, min(run.shapes[i])), (i, run.shapes[i], e)
        assert e["m"] <= TOL_M, (i, run.shapes[i], e)
        assert e["w_violations"] == 0, (i, run.shapes[i], e)
        if run.param == "f32" and run.compute == "f32":
            assert e["w"] <= TOL_W["f32"], (i, run.shapes[i], e)
    return worst


def test_toy_workload_fp32():
    w = workloads.get("toy")
    ms = make_matrix_set(w, "cuda")
    run = LibRun(w.shapes, param="f32", grad="f32", compute="f32")
    init = []
    for i in range(len(w.shapes)):
        Wi, Gi, Mi = ms.view(ms.W, i), ms.view(ms.G, i), ms.view(ms.M, i)
        run.set(i, W=Wi, G=Gi, M=Mi)
        init.append((Wi.double().cpu().numpy(), Gi.double().cpu().numpy(), Mi.double().cpu().numpy()))
    run.step(lr=w.lr, mu=w.mu, nesterov=w.nesterov)
    torch.cuda.synchronize()
    worst = _check_all(run, init, lr=w.lr, mu=w.mu, nesterov=w.nesterov)
    assert run.status() == 0
    print("toy worst", worst)


@pytest.mark.parametrize("compute", ["f32", "bf16"])
def test_golden_tiny_step(compute):
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_step.json")))
    h = gold["hyper"]
    shapes = [tuple(c["shape"]) for c in gold["cases"]]
    run = LibRun(shapes, param="f32", grad="f32", compute=compute)
    for i, c in enumerate(gold["cases"]):
        run.set(i, W=torch.tensor(c["W"], dtype=torch.float32), G=torch.tensor(c["G"], dtype=torch.float32),
                M=torch.tensor(c["M"], dtype=torch.float32))
    run.step(lr=h["lr"], mu=h["mu"], nesterov=h["nesterov"])
    torch.cuda.synchronize()
    for i, c in enumerate(gold["cases"]):
        X = run.update(i).cpu().numpy().astype(np.float64)
        Xr = np.array(c["X"])
        assert np.linalg.norm(X - Xr) / np.linalg.norm(Xr) <= tol_x(compute, min(shapes[i])), (i, compute)
        W = run.host(run.W, i)
        Wr = np.array(c["W_new"])
        r_, c_ = shapes[i]
        assert weight_rounding_violations(W, Wr, np.array(c["W"]), X, Xr, h["lr"] * ref.update_scale(r_, c_), "f32") == 0
        if compute == "f32":
            assert np.linalg.norm(W - Wr) / np.linalg.norm(Wr) <= 1e-6


@pytest.mark.parametrize("epilogue_ax", [False, True], ids=["P_X", "aX_epilogue"])
@pytest.mark.parametrize("compute", ["bf16", "f32"])
def test_ragged_shapes(compute, epilogue_ax):
    """Both forms of the quintic step: X' = P X with P = aI + bA + cA^2, and
    X' = aX + (bA + cA^2) X with the a*X term in the last product's epilogue."""
    prm = "bf16" if compute == "bf16" else "f32"
    run = LibRun(RAGGED, param=prm, grad=prm, compute=compute, epilogue_ax=epilogue_ax)
    init = _fill(run, 500, grad_std=1e-3 if compute == "bf16" else 1.0, w_std=0.02 if compute == "bf16" else 1.0,
                 m_std=1e-3)
    run.step()
    torch.cuda.synchronize()
    worst = _check_all(run, init)
    assert run.status() == 0
    print(compute, "worst", worst)


@pytest.mark.parametrize("ns_steps", [0, 1, 2, 3])
@pytest.mark.parametrize("compute", ["bf16", "f32"])
def test_ns_step_counts(ns_steps, compute):
    shapes = [(200, 300), (300, 200), (64, 64)]
    prm = "bf16" if compute == "bf16" else "f32"
    run = LibRun(shapes, param=prm, grad=prm, compute=compute, ns_steps=ns_steps)
    init = _fill(run, 900 + ns_steps)
    run.step()
    torch.cuda.synchronize()
    _check_all(run, init, ns_steps=ns_steps)


def test_per_step_coeffs_and_heavy_ball():
    coeffs = [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.0, -1.5, 0.5)]
    shapes = [(256, 512), (512, 256)]
    for compute in ("bf16", "f32"):
        run = LibRun(shapes, param="f32", grad="f32", compute=compute, ns_steps=3, coeffs=coeffs)
        init = _fill(run, 1200, m_std=1e-3)
        run.step(lr=0.05, mu=0.9, nesterov=False)
        torch.cuda.synchronize()
        for i, (W0, G, M0) in enumerate(init):
            e = compare(run, i, W0, G, M0, compute=compute, param="f32", lr=0.05, mu=0.9, nesterov=False,
                        ns_steps=3, coeffs=coeffs)
            assert e["x"] <= TOL_X[compute] and e["m"] <= TOL_M, (compute, i, e)


@pytest.mark.parametrize("param,grad", [("f32", "bf16"), ("bf16", "f32")])
def test_mixed_storage_dtypes(param, grad):
    shapes = [(384, 640), (640, 384)]
    run = LibRun(shapes, param=param, grad=grad, compute="bf16")
    init = _fill(run, 1300)
    run.step()
    torch.cuda.synchronize()
    _check_all(run, init)


def test_zero_gradient_leaves_weights():
    shapes = [(128, 256), (300, 100)]
    for compute in ("bf16", "f32"):
        prm = "bf16" if compute == "bf16" else "f32"
        run = LibRun(shapes, param=prm, grad=prm, compute=compute)
        for i, (r, c) in enumerate(shapes):
            run.set(i, W=random_matrix(r, c, 7 + i, 0.02, "cuda", prm))
        W0 = run.W.clone()
        run.step()
        torch.cuda.synchronize()
        assert torch.equal(run.W, W0)
        assert run.status() == 0
        for i in range(len(shapes)):
            assert torch.count_nonzero(run.update(i)) == 0


def _state(run):
    return run.W.clone(), run.M.clone()


def test_run_to_run_determinism_and_batch_invariance():
    shapes = [(300, 700), (700, 300), (512, 512)]
    a = LibRun(shapes)
    _fill(a, 1400, m_std=1e-3)
    W0, M0, G0 = a.W.clone(), a.M.clone(), a.G.clone()
    a.step()
    Wa, Ma = _state(a)
    # same state again: bitwise identical
    a.W.copy_(W0)
    a.M.copy_(M0)
    a.step()
    assert torch.equal(a.W, Wa) and torch.equal(a.M, Ma)
    # each matrix alone in its own plan: bitwise identical to the batched result
    for i, shp in enumerate(shapes):
        b = LibRun([shp])
        b.set(0, W=a.view(W0, i), G=a.view(G0, i), M=a.view(M0, i))
        b.step()
        assert torch.equal(b.view(b.W, 0), a.view(Wa, i)), i
        assert torch.equal(b.view(b.M, 0), a.view(Ma, i)), i


def test_resume_from_copied_state():
    # three steps straight through == one step, copy W and M out, new plan, two more steps
    shapes = [(256, 640), (640, 256)]
    grads = [[random_matrix(r, c, 1500 + 10 * k + i, 1e-3, "cuda", "bf16") for i, (r, c) in enumerate(shapes)]
             for k in range(3)]
    a = LibRun(shapes, capture=False)
    _fill(a, 1600)
    W0, M0 = a.W.clone(), a.M.clone()
    for k in range(3):
        for i in range(len(shapes)):
            a.set(i, G=grads[k][i])
        a.step()
    b = LibRun(shapes, capture=False)
    b.W.copy_(W0)
    b.M.copy_(M0)
    for i in range(len(shapes)):
        b.set(i, G=grads[0][i])
    b.step()
    Wc, Mc = b.W.clone(), b.M.clone()
    del b
    c = LibRun(shapes, capture=False)
    c.W.copy_(Wc)
    c.M.copy_(Mc)
    for k in (1, 2):
        for i in range(len(shapes)):
            c.set(i, G=grads[k][i])
        c.step()
    assert torch.equal(a.W, c.W) and torch.equal(a.M, c.M)


def test_nonfinite_norm_sets_status_bit():
    run = LibRun([(64, 128)], param="f32", grad="f32", compute="f32")
    G = torch.zeros(64, 128)
    G[3, 5] = float("inf")
    run.set(0, G=G)
    run.step()
    bits = run.status()
    assert bits & dm.DEV_NONFINITE_NORM
    assert run.status() == 0  # cleared by the read


def test_bounded_wait_gives_up_and_reports():
    scratch = torch.zeros(64, dtype=torch.int32, device="cuda")
    bits = dm.dmuon_selftest_wait_timeout(scratch.data_ptr(), 20_000_000, torch.cuda.current_stream().cuda_stream)
    assert bits & dm.DEV_WAIT_TIMEOUT
    # the context is still usable
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0


def test_launch_count_per_step():
    shapes = [(256, 512), (512, 256), (128, 128)]
    run = LibRun(shapes)
    d = run.muon.plan.describe()
    # (256, 512) runs in 256-wide tiles and (128, 128) in 128-wide ones: two chunks of 3 x 5 launches
    assert d["chunks"] == 2
    c0 = run.muon.plan.launch_count()
    run.step()
    assert run.muon.plan.launch_count() - c0 == len(d["launches"]) == 2 + 2 * 3 * 5


def test_pointer_sets_resident_and_replaced():
    """Steps that alternate among five gradient buffers (more than the four
    pointer tables a plan keeps on the device, so tables are reused and
    replaced) equal, bit for bit, steps that copy the same gradients into one
    fixed buffer."""
    shapes = [(300, 700), (700, 300), (256, 256)]
    a = LibRun(shapes, capture=False)
    b = LibRun(shapes, capture=False)
    _fill(a, 7000, m_std=1e-3)
    b.W.copy_(a.W)
    b.M.copy_(a.M)
    grads = []
    for k in range(5):
        g = torch.empty_like(a.G)
        for i, (r, c) in enumerate(shapes):
            o = a.offs[i]
            g[o:o + r * c].copy_(random_matrix(r, c, 7100 + 10 * k + i, 1e-3, "cuda", "bf16").reshape(-1))
        grads.append(g)
    stream = torch.cuda.current_stream().cuda_stream
    for k in [0, 1, 0, 1, 2, 3, 4, 0, 1, 2]:
        a.muon.plan.step(a.ptrs(a.W), a.ptrs(grads[k]), a.ptrs(a.M), 0.02, 0.95, True, stream)
        b.G.copy_(grads[k])
        b.step()
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(a.W, b.W) and torch.equal(a.M, b.M)


def test_weight_sets_replaced_store_through_their_own_maps():
    """Six weight/momentum replicas stepped in turn through one plan. That is
    more pointer sets than the four a plan keeps on the device, so slots are
    refilled with the tensor maps of other weight buffers. Each replica's
    matrices must equal, bit for bit, the same steps run through one fixed
    buffer. Every buffer stays allocated: a map left over from another set
    would write into a live buffer and show up here as a mismatch."""
    shapes = [(520, 1000), (1000, 520), (256, 256)]  # row pitches of 16-byte multiples: box stores
    a = LibRun(shapes, capture=False)
    b = LibRun(shapes, capture=False)
    _fill(a, 7300, m_std=1e-3)
    Ws, Ms = [], []
    for k in range(6):
        W, M = torch.zeros_like(a.W), torch.zeros_like(a.M)
        for i, (r, c) in enumerate(shapes):
            a.view(W, i).copy_(random_matrix(r, c, 7400 + 10 * k + i, 0.02, "cuda", "bf16"))
            a.view(M, i).copy_(random_matrix(r, c, 7500 + 10 * k + i, 1e-3, "cuda", "f32"))
        Ws.append(W)
        Ms.append(M)
    Wb, Mb = [w.clone() for w in Ws], [m.clone() for m in Ms]
    b.G.copy_(a.G)
    stream = torch.cuda.current_stream().cuda_stream
    for k in [0, 1, 2, 3, 4, 5, 0, 1, 4, 2, 5, 3]:
        a.muon.plan.step(a.ptrs(Ws[k]), a.ptrs(a.G), a.ptrs(Ms[k]), 0.02, 0.95, True, stream)
        b.W.copy_(Wb[k])
        b.M.copy_(Mb[k])
        b.step()
        Wb[k].copy_(b.W)
        Mb[k].copy_(b.M)
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    for k in range(6):
        for i in range(len(shapes)):
            assert torch.equal(a.view(Ws[k], i), a.view(Wb[k], i)), (k, i)
            assert torch.equal(a.view(Ms[k], i), a.view(Mb[k], i)), (k, i)


@pytest.mark.parametrize("flags", ["standard", "gram", "pair", "static"])
def test_cuda_graph_replay_matches_eager(flags):
    # after one uncaptured step with the same pointers, dmuon_step records no host copies and can be
    # captured; two graph replays must equal two eager steps bit for bit (the tile-claim counters
    # of each launch are left at zero by the launch itself, so replays claim from zero again)
    shapes = [(512, 1024), (1024, 512), (256, 256)]
    kw = {"gram_ns": flags == "gram", "pair": flags == "pair", "capture": False,
          "flags": dm.FLAG_STATIC_TILES if flags == "static" else 0}
    a = LibRun(shapes, **kw)
    _fill(a, 6000, m_std=1e-3)
    W0, M0 = a.W.clone(), a.M.clone()
    a.step()
    a.step()
    torch.cuda.synchronize()
    Wa, Ma = a.W.clone(), a.M.clone()
    a.W.copy_(W0)
    a.M.copy_(M0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        a.step()  # warm-up on the capture stream: uploads nothing new
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    a.W.copy_(W0)
    a.M.copy_(M0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        a.muon.plan.step(a.ptrs(a.W), a.ptrs(a.G), a.ptrs(a.M), 0.02, 0.95, True, s.cuda_stream)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a.W, Wa) and torch.equal(a.M, Ma)
