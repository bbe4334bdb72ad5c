"""The no-allocation entry point against the regular, workspace-based step.

dmuon_momentum_norm_noalloc serves callers that cannot allocate device memory
when they update their weights (a framework whose allocator already holds the
whole GPU, or a plugin that is handed only the tensors it must update): it
runs the momentum and normalisation pass of one matrix with its reduction
scratch in a static device array of the library. Here it must give the same
momentum and the same normalised matrix s*U as dmuon_step (planned with
ns_steps = 0, whose captured update is exactly s*U), on two calls in a row, so
that whatever the first call leaves in the shared array cannot leak into the
second. This file is collected last on purpose.
"""

import pytest
import torch

from matrix_optimizer_update_gb300 import dmuon as dm
from matrix_optimizer_update_gb300.inputs import random_matrix

from helpers import TOL_M, TOL_X, LibRun, rel

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(300, 700), (700, 300), (1024, 4096), (129, 257)])
def test_noalloc_pass_matches_dmuon_step_twice(shape, dtype):
    r, c = shape
    m, n = min(r, c), max(r, c)
    u_ld = (n + 7) // 8 * 8
    stream = torch.cuda.current_stream().cuda_stream
    run = LibRun([shape], param=dtype, grad=dtype, compute=dtype, ns_steps=0)
    M0 = random_matrix(r, c, 4100, 1e-3, "cuda", "f32")
    run.set(0, M=M0)
    M_na = M0.clone()
    u = torch.empty(m, u_ld, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32, device="cuda")
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    for call in range(2):
        G = random_matrix(r, c, 4200 + call, 1e-3, "cuda", dtype)
        run.set(0, G=G)
        run.step(lr=0.02, mu=0.95, nesterov=True)
        x_step = run.update(0).double().cpu().numpy()  # s * U in W's orientation
        dm.dmuon_momentum_norm_noalloc(G.data_ptr(), M_na.data_ptr(), u.data_ptr(), s.data_ptr(), r, c,
                                       dtype, dtype, 0.95, True, 1e-7, stream)
        torch.cuda.synchronize()
        U = u[:, :n].double()
        if r > c:
            U = U.t()
        x_na = (float(s.item()) * U).cpu().numpy()
        assert rel(x_na, x_step) <= TOL_X["f32"], (call, rel(x_na, x_step))
        assert rel(M_na.double().cpu().numpy(), run.host(run.M, 0)) <= TOL_M, call


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
