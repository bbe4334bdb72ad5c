"""GPU parity of the AdamW step (dmuon_adamw_flat) against the fp64 oracle,
over several steps, on a ragged buffer (not a multiple of the 8-element
vector width)."""

import numpy as np
import pytest
import torch

from matrix_optimizer_update_gb300 import dmuon as dm
from oracle.adamw_ref import adamw_step

from helpers import storage_ulp

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pdt,gdt", [("f32", "f32"), ("bf16", "bf16"), ("f32", "bf16")])
@pytest.mark.parametrize("n", [1_000_003, 5])
def test_adamw_matches_oracle(pdt, gdt, n):
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}
    gen = torch.Generator(device="cuda")
    gen.manual_seed(n + len(pdt))
    p = (torch.randn(n, generator=gen, device="cuda") * 0.02).to(tdt[pdt])
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    pr, mr, vr = p.double().cpu().numpy(), np.zeros(n), np.zeros(n)
    stream = torch.cuda.current_stream().cuda_stream

    def f(x):
        return float(np.float32(x))

    for step in range(1, 5):
        g = (torch.randn(n, generator=gen, device="cuda") * 1e-3).to(tdt[gdt])
        p_before = p.double().cpu().numpy()
        m_prev, v_prev = mr.copy(), vr.copy()
        dm.dmuon_adamw_flat(p.data_ptr(), g.data_ptr(), m.data_ptr(), v.data_ptr(), n, pdt, gdt, lr=1e-3,
                            weight_decay=0.01, step=step, stream=stream)
        torch.cuda.synchronize()
        # the oracle steps from the parameters the GPU stored (bf16 storage rounds every step), with the
        # hyperparameters as the C ABI receives them (fp32): 1 - fp32(0.999) is not 0.001
        pr, mr, vr = adamw_step(p_before, g.double().cpu().numpy(), mr, vr, lr=f(1e-3), beta1=f(0.9), beta2=f(0.999),
                                eps=f(1e-8), weight_decay=f(0.01), step=step)
        mg, vg = m.double().cpu().numpy(), v.double().cpu().numpy()
        gd = g.double().cpu().numpy()
        # fp32 blend of two terms: error within a few ulps of the larger term (they can cancel)
        m_terms = np.abs(f(0.9) * m_prev) + np.abs((1 - f(0.9)) * gd)
        v_terms = np.abs(f(0.999) * v_prev) + np.abs((1 - f(0.999)) * gd * gd)
        assert np.all(np.abs(mg - mr) <= 2.0 ** -21 * m_terms + 1e-30)
        assert np.all(np.abs(vg - vr) <= 2.0 ** -21 * v_terms + 1e-30)
        pg = p.double().cpu().numpy()
        # stored parameter = exact step rounded once to its storage type, up to the fp32 arithmetic:
        # the moments' own error (bounded above) carried through m / (sqrt(v)/sqrt(bc2) + eps), plus a
        # few ulps of the decay and of the update
        bc1, bc2 = 1 - f(0.9) ** step, 1 - f(0.999) ** step
        den = np.sqrt(vr) / np.sqrt(bc2) + f(1e-8)
        upd = f(1e-3) / bc1 * mr / den
        dm_max, dv_max = 2.0 ** -21 * m_terms, 2.0 ** -21 * v_terms
        dden = dv_max / (2 * np.sqrt(np.maximum(vr, 1e-300)) * np.sqrt(bc2))
        dupd = f(1e-3) / bc1 * (dm_max / den + np.abs(mr) * dden / den ** 2) + np.abs(upd) * 2.0 ** -20
        bound = 0.5 * storage_ulp(np.maximum(np.abs(pg), np.abs(pr)), pdt) + np.abs(p_before) * 2.0 ** -21 + dupd
        assert int(np.count_nonzero(np.abs(pg - pr) > bound)) == 0
        mr, vr = mg, vg  # continue from the stored moments


def test_adamw_rejects_bad_arguments():
    buf = torch.zeros(64, device="cuda")
    q = buf.data_ptr()
    with pytest.raises(dm.DmuonError):
        dm.dmuon_adamw_flat(q, q, q, q, 16, step=0)
    with pytest.raises(dm.DmuonError):
        dm.dmuon_adamw_flat(q + 4, q, q, q, 16)
