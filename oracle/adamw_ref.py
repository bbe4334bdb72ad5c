"""fp64 reference of the AdamW step for the parameters Muon does not own.

TEST INFRASTRUCTURE ONLY (tests/, bench CPU legs). The DMuon project docs
("DMuon", section "DMuon 能做什么", the Python example) hand every parameter
the predicate does not select to AdamW with its own learning rate
(``adamw_lr``); the pages give no other AdamW detail, so this is the
decoupled-weight-decay form with bias correction, written out step by step:

    p <- p * (1 - lr * wd)
    m <- beta1 * m + (1 - beta1) * g
    v <- beta2 * v + (1 - beta2) * g^2
    p <- p - (lr / (1 - beta1^t)) * m / (sqrt(v) / sqrt(1 - beta2^t) + eps)

Pinned in tests/test_adamw_pins.py against torch.optim.AdamW (float64) and
closed forms.
"""

from __future__ import annotations

import math

import numpy as np


def adamw_step(p, g, m, v, *, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1):
    """One AdamW step (t = ``step`` >= 1); returns (p, m, v) as new float64 arrays."""
    p = np.asarray(p, dtype=np.float64) * (1.0 - lr * weight_decay)
    g = np.asarray(g, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    denom = np.sqrt(v) / math.sqrt(bc2) + eps
    p = p - (lr / bc1) * m / denom
    return p, m, v
