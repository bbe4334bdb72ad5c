"""The no-allocation entry point against the regular, workspace-based step
and against the fp64 oracle.

dmuon_momentum_norm_noalloc serves callers that cannot allocate device memory
when they update their weights (a framework whose allocator already holds the
whole GPU, or a plugin that is handed only the tensors it must update): it
runs the momentum and normalisation pass of one matrix with its reduction
scratch in a static device array of the library. Here it must give the same
momentum and the same normalised matrix s*U as dmuon_step (planned with
ns_steps = 0, whose captured update is exactly s*U), and the momentum,
Nesterov look-ahead and Frobenius normalisation of the oracle, on two calls in
a row, so that whatever the first call leaves in the shared array cannot leak
into the second. A large call followed by a small ragged one checks the same
for calls of different sizes. This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

from matrix_optimizer_update_gb300 import dmuon as dm
from matrix_optimizer_update_gb300.inputs import random_matrix
from oracle import muon_ref as ref

from helpers import TOL_M, TOL_X, LibRun, rel

pytestmark = pytest.mark.gpu

# s*U against the oracle's U / (||U||_F + eps): U is stored once in the storage
# type (bf16: every element within 2^-9 relative, so the Frobenius error is at
# most 2^-9 as well), s comes from fp32 partial sums of squares.
TOL_SU = {"bf16": 2.0 ** -9 + 1e-5, "f32": 1e-5}


def noalloc_call(G, M, r, c, dtype, stream):
    m, n = min(r, c), max(r, c)
    u_ld = (n + 7) // 8 * 8
    u = torch.empty(m, u_ld, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32, device="cuda")
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    dm.dmuon_momentum_norm_noalloc(G.data_ptr(), M.data_ptr(), u.data_ptr(), s.data_ptr(), r, c, dtype, dtype,
                                   0.95, True, 1e-7, stream)
    torch.cuda.synchronize()
    U = u[:, :n].double()
    if r > c:
        U = U.t()
    return float(s.item()), U.cpu().numpy()


def oracle_pass(M0, G):
    M_new, U = ref.momentum_update(M0, G, 0.95, True)
    return M_new, U, ref.frobenius_normalize(U, 1e-7)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(300, 700), (700, 300), (1024, 4096), (129, 257)])
def test_noalloc_pass_matches_dmuon_step_and_oracle_twice(shape, dtype):
    r, c = shape
    stream = torch.cuda.current_stream().cuda_stream
    run = LibRun([shape], param=dtype, grad=dtype, compute=dtype, ns_steps=0)
    M0 = random_matrix(r, c, 4100, 1e-3, "cuda", "f32")
    run.set(0, M=M0)
    M_na = M0.clone()
    M_ref = M0.double().cpu().numpy()
    for call in range(2):
        G = random_matrix(r, c, 4200 + call, 1e-3, "cuda", dtype)
        run.set(0, G=G)
        run.step(lr=0.02, mu=0.95, nesterov=True)
        x_step = run.update(0).double().cpu().numpy()  # s * U in W's orientation
        s, U = noalloc_call(G, M_na, r, c, dtype, stream)
        x_na = s * U
        assert rel(x_na, x_step) <= TOL_X["f32"], (call, rel(x_na, x_step))
        assert rel(M_na.double().cpu().numpy(), run.host(run.M, 0)) <= TOL_M, call
        # the oracle, on the same inputs
        M_ref, _, X0 = oracle_pass(M_ref, G.double().cpu().numpy())
        assert rel(M_na.double().cpu().numpy(), M_ref) <= TOL_M, call
        assert rel(x_na, X0) <= TOL_SU[dtype], (call, rel(x_na, X0))


def test_noalloc_large_then_small_ragged():
    """A small call after a large one reads only its own partial sums."""
    stream = torch.cuda.current_stream().cuda_stream
    for (r, c), seed in (((4096, 4096), 4300), ((129, 257), 4301), ((2048, 1408), 4302), ((67, 45), 4303)):
        G = random_matrix(r, c, seed, 1e-3, "cuda", "bf16")
        M = random_matrix(r, c, seed + 50, 1e-3, "cuda", "f32")
        M0 = M.double().cpu().numpy()
        s, U = noalloc_call(G, M, r, c, "bf16", stream)
        M_ref, U_ref, X0 = oracle_pass(M0, G.double().cpu().numpy())
        s_ref = 1.0 / (np.linalg.norm(U_ref) + 1e-7)
        assert abs(s - s_ref) <= 1e-5 * s_ref, ((r, c), s, s_ref)
        assert rel(s * U, X0) <= TOL_SU["bf16"], (r, c)
        assert rel(M.double().cpu().numpy(), M_ref) <= TOL_M, (r, c)


def test_noalloc_rejects_too_large_and_bad_arguments():
    stream = torch.cuda.current_stream().cuda_stream
    buf = torch.empty(64, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    with pytest.raises(dm.DmuonError) as e:
        dm.dmuon_momentum_norm_noalloc(p, p, p, p, 1 << 20, 1 << 10, stream=stream)  # 16384 x 8 tiles: too many
    assert e.value.status == dm.ERR_UNSUPPORTED and "static scratch" in str(e.value)
    with pytest.raises(dm.DmuonError) as e:
        dm.dmuon_momentum_norm_noalloc(0, p, p, p, 4, 4, stream=stream)
    assert e.value.status == dm.ERR_INVALID_ARG
