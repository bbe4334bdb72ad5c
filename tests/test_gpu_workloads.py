"""Parity on the full-size workloads, in the plan and launch configuration the
benchmark times: the whole matrix set steps on the GPU; sampled matrices are
checked one by one against the fp64 oracle (X within 2e-2, stored bf16 weights
within 1e-3 of the oracle's rounded weights, momentum within 1e-6), and every
matrix is checked for properties that hold at any size."""

import numpy as np
import pytest
import torch

from matrix_optimizer_update_gb300 import dmuon as dm
from matrix_optimizer_update_gb300 import workloads as wl
from matrix_optimizer_update_gb300.inputs import expert_scales, make_matrix_set
from oracle import muon_ref as ref

from helpers import TOL_M, TOL_W, TOL_X, rel, weight_rounding_violations

pytestmark = pytest.mark.gpu


def sample_indices(w, full_last_layer=False):
    mats = list(w.matrices())
    L = w.layers
    if w.experts:
        # layer 0 attention, plus 16 seeded experts including the smallest- and largest-scale ones
        idx = [i for i, (layer, role, r, c, e) in enumerate(mats) if layer == 0 and e < 0]
        sc = expert_scales(w)
        lo = np.unravel_index(np.argmin(sc), sc.shape)
        hi = np.unravel_index(np.argmax(sc), sc.shape)
        rng = np.random.default_rng(77)
        picks = {tuple(lo), tuple(hi)}
        while len(picks) < 16:
            picks.add((int(rng.integers(L)), int(rng.integers(w.experts))))
        roles = ["gate", "up", "down"]
        for k, (layer, e) in enumerate(sorted(picks)):
            role = roles[k % 3]
            idx += [i for i, (la, ro, r, c, ee) in enumerate(mats) if la == layer and ee == e and ro == role]
        return sorted(set(idx))
    if w.name == "llama-3.1-8b" and not full_last_layer:
        # the variant forms: layer 0 and two matrices of the last layer (the standard form checks every
        # matrix of both layers)
        last = [i for i, m in enumerate(mats) if m[0] == L - 1 and m[1] in ("k", "gate")]
        return [i for i, m in enumerate(mats) if m[0] == 0] + last
    return [i for i, m in enumerate(mats) if m[0] in (0, L - 1)]


# one_sm: one-SM tiles everywhere instead of the default two-SM pairs where they fill the short side
@pytest.mark.parametrize("name,gram,one_sm,ax", [("qwen2.5-1.5b", False, False, False),
                                                 ("llama-3.2-3b", False, False, False),
                                                 ("llama-3.1-8b", False, False, False),
                                                 ("moe-16x64", False, False, False),
                                                 ("llama-3.1-8b", True, False, False),
                                                 ("moe-16x64", True, False, False),
                                                 ("llama-3.1-8b", False, True, False),
                                                 ("llama-3.1-8b", False, False, True)])
def test_workload_parity(name, gram, one_sm, ax):
    w = wl.get(name)
    ms = make_matrix_set(w, "cuda")
    idx = sample_indices(w, full_last_layer=not (gram or one_sm or ax))
    before = {i: (ms.view(ms.W, i).double().cpu().numpy(), ms.view(ms.G, i).double().cpu().numpy(),
                  ms.view(ms.M, i).double().cpu().numpy()) for i in idx}
    muon = dm.Muon.create(w.shapes, ns_steps=w.ns_steps, coeffs=w.coeffs, eps=w.eps, param=w.param_dtype,
                          grad=w.grad_dtype, compute=w.compute,
                          flags=dm.FLAG_CAPTURE_UPDATE | (dm.FLAG_GRAM_NS if gram else 0)
                          | (dm.FLAG_ONE_SM_TILES if one_sm else 0) | (dm.FLAG_EPILOGUE_AX if ax else 0))
    stream = torch.cuda.current_stream().cuda_stream
    muon.plan.step(ms.ptrs(ms.W), ms.ptrs(ms.G), ms.ptrs(ms.M), w.lr, w.mu, w.nesterov, stream)
    torch.cuda.synchronize()
    assert muon.plan.read_device_status(stream) == 0

    # properties of every matrix: finite weights, and ||X||_F / sqrt(m) inside the band
    # [0.68, 1.21] that the quintic maps every normalised singular value >= 3e-3 into
    x = torch.empty(max(r * c for r, c in w.shapes), dtype=torch.float32, device="cuda")
    for i, (r, c) in enumerate(w.shapes):
        assert bool(torch.isfinite(ms.view(ms.W, i)).all()), i
        muon.plan.read_update(i, x.data_ptr(), stream)
        nrm = float(torch.linalg.vector_norm(x[: r * c])) / np.sqrt(min(r, c))
        assert 0.68 <= nrm <= 1.21, (i, r, c, nrm)

    # The default form keeps its stored weights at least 5 % under the 1e-3 bar on every workload
    # (measured worst: MoE 9.1e-4; one-SM tiles give the same bits); the opt-in forms are held to the
    # bar itself.
    w_bar = TOL_W[w.param_dtype] * (0.95 if not (gram or ax) else 1.0)
    worst = {"x": 0.0, "w": 0.0, "m": 0.0, "worst_w_matrix": None}
    for i in idx:
        r, c = w.shapes[i]
        W0, G, M0 = before[i]
        Wr, Mr, Xr = ref.muon_step(W0, G, M0, lr=w.lr, mu=w.mu, nesterov=w.nesterov, ns_steps=w.ns_steps,
                                   coeffs=w.coeffs, eps=w.eps)
        muon.plan.read_update(i, x.data_ptr(), stream)
        Xg = x[: r * c].view(r, c).double().cpu().numpy()
        Wg = ms.view(ms.W, i).double().cpu().numpy()
        Mg = ms.view(ms.M, i).double().cpu().numpy()
        ex = rel(Xg, Xr)
        ew = float(np.linalg.norm(Wg - ref.round_to_dtype(Wr, w.param_dtype)) / np.linalg.norm(Wr))
        em = rel(Mg, Mr)
        if ew > worst["w"]:
            worst["worst_w_matrix"] = (i, r, c)
        worst.update(x=max(worst["x"], ex), w=max(worst["w"], ew), m=max(worst["m"], em))
        assert ex <= TOL_X[w.compute], (i, r, c, ex)
        assert ew <= w_bar, (i, r, c, ew, w_bar)
        assert em <= TOL_M, (i, r, c, em)
        assert weight_rounding_violations(Wg, Wr, W0, Xg, Xr, w.lr * ref.update_scale(r, c), w.param_dtype) == 0
    print(name, "gram" if gram else "standard", "one-SM" if one_sm else "", "aX-epilogue" if ax else "", "sampled",
          len(idx), "worst", worst)
