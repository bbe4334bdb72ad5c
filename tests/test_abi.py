"""C-ABI checks that need no GPU: the library loads, exports every function
include/dmuon.h declares, and the host planner validates, buckets and
counts tiles as stated."""

import os
import re
import subprocess
import sys

import numpy as np
import pytest

from matrix_optimizer_update_gb300 import dmuon as dm
from matrix_optimizer_update_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dmuon.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dmuon_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(dm.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = dm.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert dm.dmuon_version() >= 100


def test_invalid_arguments_are_rejected_on_the_host():
    with pytest.raises(dm.DmuonError) as e:
        dm.dmuon_plan([], 5)
    assert e.value.status == dm.ERR_INVALID_ARG
    for bad in ([(0, 4)], [(4, -1)], [(1 << 21, 4)], [(65536, 65536)]):
        with pytest.raises(dm.DmuonError) as e:
            dm.dmuon_plan(bad, 5)
        assert e.value.status == dm.ERR_INVALID_ARG
    with pytest.raises(dm.DmuonError) as e:
        dm.dmuon_plan([(4, 4)], 17)
    assert e.value.status == dm.ERR_INVALID_ARG
    with pytest.raises(dm.DmuonError) as e:
        dm.dmuon_plan([(4, 4)], 3, coeffs=[(1, 2, 3), (1, 2, 3)])
    assert e.value.status == dm.ERR_INVALID_ARG
    with pytest.raises(dm.DmuonError) as e:
        dm.dmuon_plan([(4, 4)], 3, eps=-1.0)
    assert e.value.status == dm.ERR_INVALID_ARG
    with pytest.raises(dm.DmuonError) as e:
        dm.dmuon_plan([(4, 4)], 3, flags=0x100)
    assert e.value.status == dm.ERR_UNSUPPORTED
    for both in (dm.FLAG_PAIR_TILES, dm.FLAG_TUNE):
        with pytest.raises(dm.DmuonError) as e:
            dm.dmuon_plan([(4, 4)], 3, flags=dm.FLAG_ONE_SM_TILES | both)
        assert e.value.status == dm.ERR_INVALID_ARG


def test_step_before_bind_is_refused():
    p = dm.dmuon_plan([(8, 16)], 5)
    with pytest.raises(dm.DmuonError) as e:
        p.step([16], [32], [48], 0.02, 0.95, True, 0)
    assert e.value.status == dm.ERR_NOT_BOUND
    with pytest.raises(dm.DmuonError) as e:
        p.bind(0, 1 << 20, 0)
    assert e.value.status == dm.ERR_WORKSPACE
    with pytest.raises(dm.DmuonError) as e:
        p.bind(1024 * 7 + 16, 1 << 40, 0)  # misaligned
    assert e.value.status == dm.ERR_WORKSPACE
    with pytest.raises(dm.DmuonError) as e:
        p.bind(1024 * 1024, 16, 0)  # too small
    assert e.value.status == dm.ERR_WORKSPACE
    with pytest.raises(dm.DmuonError) as e:
        p.read_update(0, 1024, 0)
    assert e.value.status == dm.ERR_UNSUPPORTED


def test_failed_bind_leaves_the_plan_unbound(monkeypatch):
    # the host-side failure hook fires before any CUDA call: no GPU needed
    p = dm.dmuon_plan([(8, 16)], 5)
    monkeypatch.setenv("DMUON_TEST_FAIL", "bind_check")
    with pytest.raises(dm.DmuonError) as e:
        p.bind(1 << 30, p.workspace_bytes(), 0)
    assert e.value.status == dm.ERR_CUDA and "injected failure" in str(e.value)
    monkeypatch.delenv("DMUON_TEST_FAIL")
    with pytest.raises(dm.DmuonError) as e:
        p.step([16], [32], [48], 0.02, 0.95, True, 0)
    assert e.value.status == dm.ERR_NOT_BOUND


def test_log_switch_writes_plan_lines_to_stderr():
    code = ("from matrix_optimizer_update_gb300 import dmuon as dm; "
            "p = dm.dmuon_plan([(256, 384), (384, 256), (64, 64)], 5); p.destroy()")
    env = dict(os.environ, DMUON_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT, timeout=120)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stderr.splitlines() if x.startswith("[dmuon]")]
    assert any("plan" in x and "3 matrices" in x for x in lines), r.stderr
    assert sum(x.startswith("[dmuon]   bucket") for x in lines) == 2, r.stderr
    env.pop("DMUON_LOG")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT, timeout=120)
    assert r.returncode == 0 and "[dmuon]" not in r.stderr


def cdiv(a, b):
    return -(-a // b)


def brute_tiles(m, n, bm, bn_sym, bn_gemm):
    # symmetric products: row block ti's tiles start at its diagonal block, columns ti*bm + tj*bn_sym..,
    # as long as they start inside the matrix
    gram = sum(1 for ti in range(cdiv(m, bm)) for tj in range(cdiv(m, bn_sym)) if ti * bm + tj * bn_sym < m)
    gemm = cdiv(m, bm) * cdiv(n, bn_gemm)
    return gram, gemm


@pytest.mark.parametrize("name", ["toy", "qwen2.5-1.5b", "llama-3.2-3b", "llama-3.1-8b", "moe-16x64"])
def test_plan_buckets_tiles_and_work(name):
    w = wl.get(name)
    p = dm.dmuon_plan(w.shapes, w.ns_steps, w.coeffs, w.eps, w.param_dtype, w.grad_dtype, w.compute)
    d = p.describe()
    bm = d["tile"][0]
    # buckets: one per distinct (short, long) shape, counts and transposed counts add up
    want = {}
    for r, c in w.shapes:
        k = (min(r, c), max(r, c))
        cnt, tr = want.get(k, (0, 0))
        want[k] = (cnt + 1, tr + (r > c))
    got = {(b["m"], b["n"]): (b["count"], b["transposed"]) for b in d["buckets"]}
    assert got == want
    # tile counts: upper-triangle tiles for the symmetric products, full grid for the gemm; pair tiles
    # are 256 rows high
    def rows(b):
        return 256 if b["pair"] else bm

    g_tot = sum(b["count"] * brute_tiles(b["m"], b["n"], rows(b), b["bn_sym"], b["bn_gemm"])[0] for b in d["buckets"])
    m_tot = sum(b["count"] * brute_tiles(b["m"], b["n"], rows(b), b["bn_sym"], b["bn_gemm"])[1] for b in d["buckets"])
    for b in d["buckets"]:
        if w.compute == "bf16":
            # 256-wide tiles unless 1.4x their count exceeds the count of 128-wide ones
            sym = {bn: brute_tiles(b["m"], b["n"], bm, bn, bn)[0] for bn in (128, 256)}
            gemm = {bn: brute_tiles(b["m"], b["n"], bm, bn, bn)[1] for bn in (128, 256)}
            assert b["bn_sym"] == (256 if 1.4 * sym[256] <= sym[128] else 128), b
            assert b["bn_gemm"] == (256 if 1.4 * gemm[256] <= gemm[128] else 128), b
            # two-SM pairs by default where 256 x 256 tiles fill a short side of at least 1024
            assert b["pair"] == (b["m"] % 256 == 0 and b["m"] >= 1024 and b["bn_sym"] == b["bn_gemm"] == 256), b
        else:
            assert not b["pair"], b
    assert sum(c["gram"] for c in d["lists"]) == g_tot
    assert sum(c["poly"] for c in d["lists"]) == g_tot
    assert sum(c["gemm"] for c in d["lists"]) == m_tot
    # launches per step and the algorithmic work the profiler attributes to them
    assert len(d["launches"]) == 2 + 3 * w.ns_steps * d["chunks"]  # momentum, norm, 3 per step and chunk
    # every launch of a chunk shares the chunk's tile widths
    assert [L["kind"] for L in d["launches"][:2]] == [dm.KIND_MOMENTUM, dm.KIND_NORM]
    for L in d["launches"][2:]:
        assert L["bn"] in ((128, 256) if w.compute == "bf16" else (32,))  # fp32: 32 x 32 SIMT tiles
    work = {}
    for L in d["launches"]:
        work[L["kind"]] = work.get(L["kind"], 0.0) + L["work"]
    flops = sum(wl.ns_flops(r, c, w.ns_steps) for r, c in w.shapes)
    assert abs(work[dm.KIND_GRAM] + work[dm.KIND_POLY] + work[dm.KIND_GEMM] - flops) / flops < 1e-12
    xel = 2 if w.compute == "bf16" else 4
    gb = 2 if w.grad_dtype == "bf16" else 4
    assert work[dm.KIND_MOMENTUM] == sum(r * c for r, c in w.shapes) * (gb + 8 + xel)
    assert p.workspace_bytes() > 0


def test_workspace_holds_weight_maps_only_where_the_last_step_stores_through_them():
    """With bf16 weights on the tensor-core path, the workspace holds a
    128-byte TMA map of every weight matrix for each of the four resident
    pointer sets (the last step stores its updated W boxes through them).
    fp32 weights, fp32 compute and ns_steps = 0 need none."""
    shapes = [(520, 1000), (1000, 520), (256, 256), (4096, 1024), (3000, 100)]
    align = 1024  # workspace regions start on 1024-byte boundaries

    def ws(ns_steps=5, **kw):
        return dm.dmuon_plan(shapes, ns_steps, **kw).workspace_bytes()

    grow = ws(param="bf16") - ws(param="f32")
    assert 4 * len(shapes) * 128 <= grow < 4 * len(shapes) * 128 + align
    assert ws(param="bf16", compute="f32") == ws(param="f32", compute="f32")
    assert ws(0, param="bf16") == ws(0, param="f32")


MAX_BUCKETS_PER_LAUNCH = 7


def test_many_buckets_split_into_chunks():
    """Buckets with the same iteration form and tile widths share a launch, at
    most seven to a launch (the bucket descriptors fill the 4 KB of launch
    parameters)."""
    shapes = [(16 * (k + 1), 256) for k in range(19)]
    p = dm.dmuon_plan(shapes, 2)
    d = p.describe()
    assert len(d["buckets"]) == 19
    groups = {}
    for b in d["buckets"]:
        key = (b["bn_sym"], b["bn_gemm"])
        groups[key] = groups.get(key, 0) + 1
    want = sum(cdiv(n, MAX_BUCKETS_PER_LAUNCH) for n in groups.values())
    assert len(groups) == 2 and d["chunks"] == want == 4
    assert len(d["launches"]) == 2 + 3 * 2 * want


def test_ns_steps_zero_plan():
    p = dm.dmuon_plan([(64, 128), (128, 64)], 0)
    kinds = [L["kind"] for L in p.describe()["launches"]]
    assert kinds == [dm.KIND_MOMENTUM, dm.KIND_NORM, dm.KIND_UPDATE0]


def test_plan_is_deterministic():
    w = wl.get("moe-16x64")
    a = dm.dmuon_plan(w.shapes, 5).describe()
    b = dm.dmuon_plan(w.shapes, 5).describe()
    assert a == b


def test_gram_form_plan_launches_and_work():
    w = wl.get("llama-3.1-8b")
    S = w.ns_steps
    p = dm.dmuon_plan(w.shapes, S, flags=dm.FLAG_GRAM_NS)
    d = p.describe()
    forms = {(b["m"], b["n"]): b["form"] for b in d["buckets"]}
    assert forms == {(4096, 14336): "gram", (4096, 4096): "standard", (1024, 4096): "gram"}
    std_chunks, gram_chunks = 1, 1
    assert len(d["launches"]) == 2 + 3 * S * std_chunks + (4 * S - 1) * gram_chunks
    # executed work: standard buckets as before; Gram buckets: X X^T once, S polys, (S-1) Q products,
    # 2(S-1) G products (symmetric products counted once) and the final 2 m^2 n product
    want = 0.0
    for r, c in w.shapes:
        m, n = min(r, c), max(r, c)
        if n >= 2 * m:
            sym = m * m * (m + 1)
            want += m * (m + 1) * n + S * sym + (S - 1) * sym + 2 * (S - 1) * sym + 2 * m * m * n
        else:
            want += wl.ns_flops(r, c, S)
    got = sum(L["work"] for L in d["launches"] if L["kind"] not in (dm.KIND_MOMENTUM, dm.KIND_NORM))
    assert abs(got - want) / want < 1e-12
    assert got < 0.6 * sum(wl.ns_flops(r, c, S) for r, c in w.shapes)


def test_costs_need_a_tuned_plan():
    p = dm.dmuon_plan([(64, 128)], 5, flags=dm.FLAG_TUNE)
    with pytest.raises(dm.DmuonError) as e:
        p.costs()
    assert e.value.status == dm.ERR_UNSUPPORTED


@pytest.mark.parametrize("ax", [False, True])
def test_polynomial_coefficients_per_launch(ax):
    """Standard form: the step's polynomial aX + (bA + cA^2)X is formed either as
    P = aI + bA + cA^2 (a on the diagonal of the symmetric product, the last
    product with a = 0) or, with FLAG_EPILOGUE_AX, with a*X in the last
    product's epilogue. Per-step coefficients land on their own step."""
    coeffs = [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.0, -1.5, 0.5)]
    p = dm.dmuon_plan([(256, 512), (512, 256)], 3, coeffs, flags=dm.FLAG_EPILOGUE_AX if ax else 0)
    launches = p.describe()["launches"]
    for L in launches[2:]:
        a, b, c = (float(np.float32(x)) for x in coeffs[L["step"]])
        if L["kind"] == dm.KIND_POLY:
            assert (L["b"], L["c"]) == pytest.approx((b, c), rel=1e-7)
            assert L["diag"] == pytest.approx(0.0 if ax else a, rel=1e-7)
        elif L["kind"] == dm.KIND_GEMM:
            assert L["a"] == pytest.approx(a if ax else 0.0, rel=1e-7)
            assert L["diag"] == 0.0
        else:
            assert L["kind"] == dm.KIND_GRAM and L["a"] == 0.0 and L["diag"] == 0.0


@pytest.mark.parametrize("name", ["qwen2.5-1.5b", "moe-16x64"])
def test_workspace_regions_are_disjoint_and_do_not_depend_on_tiling(name):
    """The regions describe lists lie inside the workspace and do not overlap; and the layout is the
    same whatever the tile configuration (the tuner re-plans tile widths and pairs after the caller
    has sized the workspace, so nothing may move with them)."""
    w = wl.get(name)
    plans = [dm.dmuon_plan(w.shapes, w.ns_steps, flags=f)
             for f in (0, dm.FLAG_ONE_SM_TILES, dm.FLAG_TUNE, dm.FLAG_STATIC_TILES)]
    descs = [p.describe() for p in plans]
    for p, d in zip(plans, descs):
        regs = [d["regions"]["status"]] + d["regions"]["tables"] + d["regions"]["scratch"]
        regs = sorted((o, o + n) for o, n in regs)
        assert regs[0][0] >= 0 and regs[-1][1] <= p.workspace_bytes()
        for (a0, a1), (b0, b1) in zip(regs, regs[1:]):
            assert a1 <= b0, (a0, a1, b0, b1)
    assert all(d["regions"] == descs[0]["regions"] for d in descs)
    assert len({p.workspace_bytes() for p in plans}) == 1


def test_many_tile_configurations_keep_the_layout():
    # 19 buckets whose default widths differ: each could become a launch chunk of its own
    shapes = [(16 * (k + 1), 256 + 64 * k) for k in range(19)]
    a = dm.dmuon_plan(shapes, 3)
    b = dm.dmuon_plan(shapes, 3, flags=dm.FLAG_PAIR_TILES | dm.FLAG_TUNE)
    assert a.describe()["regions"] == b.describe()["regions"]
    assert a.workspace_bytes() == b.workspace_bytes()
