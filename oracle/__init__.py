"""Plain fp64 CPU oracle for the owner-side Muon update.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import anything under ``oracle/``. The
product path (the C-ABI library and its Python binding) never calls it and
shares no code with it.
"""

from .muon_ref import (  # noqa: F401
    DEFAULT_COEFFS,
    frobenius_normalize,
    momentum_update,
    muon_step,
    newton_schulz,
    newton_schulz_gram,
    orthogonalize,
    round_to_dtype,
    update_scale,
)
