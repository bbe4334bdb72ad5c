"""ctypes binding of the C ABI in include/dmuon.h.

Argument marshalling only: every step of the update runs in the library's
CUDA kernels. PyTorch is used by callers for device memory and streams; the
functions here take plain integers (device addresses, stream handles).

Loading fails loudly (``DmuonError``) when the shared library has not been
built: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import json
import os
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdmuon.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_NOT_BOUND = -5
ERR_DEVICE = -6

F32 = 0
BF16 = 1
DTYPE = {"f32": F32, "bf16": BF16}

FLAG_CAPTURE_UPDATE = 0x1
FLAG_GRAM_NS = 0x2
FLAG_TUNE = 0x4
FLAG_PAIR_TILES = 0x8
FLAG_EPILOGUE_AX = 0x10
FLAG_STATIC_TILES = 0x20
FLAG_DEBUG_CHECKS = 0x40
FLAG_ONE_SM_TILES = 0x80
DEV_NONFINITE_NORM = 0x1
DEV_WAIT_TIMEOUT = 0x2

KIND_MOMENTUM, KIND_GRAM, KIND_POLY, KIND_GEMM, KIND_UPDATE0, KIND_SYMM, KIND_NORM = range(7)
KIND_NAMES = {0: "momentum", 1: "gram", 2: "poly", 3: "gemm", 4: "update0", 5: "symm", 6: "norm"}

# every symbol include/dmuon.h declares
EXPORTS = (
    "dmuon_plan", "dmuon_plan_workspace_bytes", "dmuon_plan_bind", "dmuon_step",
    "dmuon_set_weight_events", "dmuon_read_device_status", "dmuon_read_update", "dmuon_plan_describe",
    "dmuon_profile_begin", "dmuon_profile_end", "dmuon_profile_cta_times", "dmuon_read_cta_times",
    "dmuon_plan_costs", "dmuon_launch_count",
    "dmuon_selftest_wait_timeout", "dmuon_momentum_norm_noalloc", "dmuon_assign_owners", "dmuon_adamw_flat",
    "dmuon_plan_destroy", "dmuon_last_error", "dmuon_version",
)


class DmuonError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"dmuon status {status}: {msg}")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class Dtypes(ctypes.Structure):
    _fields_ = [("param", ctypes.c_int32), ("grad", ctypes.c_int32),
                ("momentum", ctypes.c_int32), ("compute", ctypes.c_int32)]


_lib = None


def lib():
    """Load libdmuon.so (once). Raises DmuonError if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise DmuonError(ERR_CUDA, f"{LIB_PATH} is not built; run python -m matrix_optimizer_update_gb300.build")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, u32, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                  ctypes.c_float, ctypes.c_size_t)
    sig = {
        "dmuon_plan": (i32, [ctypes.POINTER(Shape), i32, i32, ctypes.POINTER(f32), i32, f32, Dtypes, u32,
                             ctypes.POINTER(vp)]),
        "dmuon_plan_workspace_bytes": (i32, [vp, ctypes.POINTER(sz)]),
        "dmuon_plan_bind": (i32, [vp, vp, sz, vp]),
        "dmuon_step": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), f32, f32, i32, vp]),
        "dmuon_set_weight_events": (i32, [vp, vp, vp]),
        "dmuon_read_device_status": (i32, [vp, vp, ctypes.POINTER(u32)]),
        "dmuon_read_update": (i32, [vp, i32, vp, vp]),
        "dmuon_plan_describe": (i32, [vp, ctypes.c_char_p, sz, ctypes.POINTER(sz)]),
        "dmuon_profile_begin": (i32, [vp, i32]),
        "dmuon_profile_end": (i32, [vp, ctypes.POINTER(i32), ctypes.POINTER(f32), ctypes.POINTER(ctypes.c_double),
                                    i32, ctypes.POINTER(i32)]),
        "dmuon_profile_cta_times": (i32, [vp, i32]),
        "dmuon_read_cta_times": (i32, [vp, i32, ctypes.POINTER(ctypes.c_uint64), i32, ctypes.POINTER(i32), vp]),
        "dmuon_plan_costs": (i32, [vp, ctypes.POINTER(ctypes.c_double), i32]),
        "dmuon_launch_count": (i32, [vp, ctypes.POINTER(i64)]),
        "dmuon_selftest_wait_timeout": (i32, [vp, i64, vp, ctypes.POINTER(u32)]),
        "dmuon_momentum_norm_noalloc": (i32, [vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, f32, vp]),
        "dmuon_assign_owners": (i32, [ctypes.POINTER(Shape), i32, i32, ctypes.POINTER(ctypes.c_double), i32,
                                      ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_double)]),
        "dmuon_adamw_flat": (i32, [vp, vp, vp, vp, i64, i32, i32, f32, f32, f32, f32, f32, i32, vp]),
        "dmuon_plan_destroy": (None, [vp]),
        "dmuon_last_error": (ctypes.c_char_p, []),
        "dmuon_version": (i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(st: int):
    if st != OK:
        raise DmuonError(st, lib().dmuon_last_error().decode())


def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * len(ptrs))()
    for i, p in enumerate(ptrs):
        arr[i] = int(p)
    return arr


def dmuon_version() -> int:
    return lib().dmuon_version()


def dmuon_plan(shapes, ns_steps=5, coeffs=(3.4445, -4.7750, 2.0315), eps=1e-7,
               param="bf16", grad="bf16", compute="bf16", flags=0) -> "Plan":
    """Build a plan (host only). ``coeffs`` is one (a, b, c) or ns_steps triples."""
    n = len(shapes)
    sh = (Shape * max(n, 1))(*[Shape(int(r), int(c)) for r, c in shapes])
    flat = []
    if coeffs is not None and len(coeffs) and isinstance(coeffs[0], (tuple, list)):
        for t in coeffs:
            flat.extend(t)
        triples = len(coeffs)
    elif coeffs is not None:
        flat = list(coeffs)
        triples = 1
    else:
        triples = 0
    cf = (ctypes.c_float * max(len(flat), 1))(*flat) if flat else None
    dt = Dtypes(DTYPE[param], DTYPE[grad], F32, DTYPE[compute])
    h = ctypes.c_void_p()
    _check(lib().dmuon_plan(sh if n else None, n, ns_steps, cf, triples, eps, dt, flags, ctypes.byref(h)))
    return Plan(h, list(shapes), ns_steps)


class Plan:
    """Owns a ``dmuon_plan_t`` handle; thin wrappers over the C calls."""

    def __init__(self, handle, shapes, ns_steps):
        self._h = handle
        self.shapes = shapes
        self.ns_steps = ns_steps
        self._ptr_cache = None

    @property
    def handle(self):
        return self._h

    def workspace_bytes(self) -> int:
        n = ctypes.c_size_t()
        _check(lib().dmuon_plan_workspace_bytes(self._h, ctypes.byref(n)))
        return n.value

    def bind(self, d_workspace: int, nbytes: int, stream: int = 0):
        _check(lib().dmuon_plan_bind(self._h, ctypes.c_void_p(d_workspace), nbytes, ctypes.c_void_p(stream)))

    def step(self, params, grads, momenta, lr, mu, nesterov, stream: int = 0):
        key = (tuple(params), tuple(grads), tuple(momenta))
        if self._ptr_cache is None or self._ptr_cache[0] != key:
            self._ptr_cache = (key, _ptr_array(params), _ptr_array(grads), _ptr_array(momenta))
        _, pa, ga, ma = self._ptr_cache
        _check(lib().dmuon_step(self._h, pa, ga, ma, float(lr), float(mu), int(bool(nesterov)),
                                ctypes.c_void_p(stream)))

    def set_weight_events(self, wait_before_write: int = 0, after_write: int = 0):
        """cudaEvent_t handles (ints, 0 = none): see dmuon_set_weight_events."""
        _check(lib().dmuon_set_weight_events(self._h, ctypes.c_void_p(wait_before_write or None),
                                             ctypes.c_void_p(after_write or None)))

    def read_device_status(self, stream: int = 0) -> int:
        b = ctypes.c_uint32()
        _check(lib().dmuon_read_device_status(self._h, ctypes.c_void_p(stream), ctypes.byref(b)))
        return b.value

    def read_update(self, mat: int, d_dst: int, stream: int = 0):
        _check(lib().dmuon_read_update(self._h, mat, ctypes.c_void_p(d_dst), ctypes.c_void_p(stream)))

    def describe(self) -> dict:
        need = ctypes.c_size_t()
        _check(lib().dmuon_plan_describe(self._h, None, 0, ctypes.byref(need)))
        buf = ctypes.create_string_buffer(need.value)
        _check(lib().dmuon_plan_describe(self._h, buf, need.value, ctypes.byref(need)))
        return json.loads(buf.value.decode())

    def profile_begin(self, max_launches: int):
        _check(lib().dmuon_profile_begin(self._h, max_launches))

    def profile_end(self, cap: int):
        kinds = (ctypes.c_int32 * cap)()
        ms = (ctypes.c_float * cap)()
        work = (ctypes.c_double * cap)()
        n = ctypes.c_int32()
        _check(lib().dmuon_profile_end(self._h, kinds, ms, work, cap, ctypes.byref(n)))
        k = min(n.value, cap)
        return [(kinds[i], ms[i], work[i]) for i in range(k)]

    def profile_cta_times(self, enable: bool = True):
        _check(lib().dmuon_profile_cta_times(self._h, int(bool(enable))))

    def read_cta_times(self, launch: int, stream: int = 0):
        """[(start_ns, end_ns)] per CTA of launch `launch` of the last recorded step."""
        n = ctypes.c_int32()
        _check(lib().dmuon_read_cta_times(self._h, launch, None, 0, ctypes.byref(n), ctypes.c_void_p(stream)))
        if n.value == 0:
            return []
        buf = (ctypes.c_uint64 * (2 * n.value))()
        _check(lib().dmuon_read_cta_times(self._h, launch, buf, n.value, ctypes.byref(n), ctypes.c_void_p(stream)))
        return [(buf[2 * i], buf[2 * i + 1]) for i in range(n.value)]

    def costs(self):
        """Measured per-matrix cost (ms) of a tuned plan."""
        n = len(self.shapes)
        out = (ctypes.c_double * n)()
        _check(lib().dmuon_plan_costs(self._h, out, n))
        return list(out)

    def launch_count(self) -> int:
        c = ctypes.c_int64()
        _check(lib().dmuon_launch_count(self._h, ctypes.byref(c)))
        return c.value

    def destroy(self):
        if self._h is not None and self._h.value:
            lib().dmuon_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def dmuon_selftest_wait_timeout(d_scratch: int, limit_ns: int, stream: int = 0) -> int:
    b = ctypes.c_uint32()
    _check(lib().dmuon_selftest_wait_timeout(ctypes.c_void_p(d_scratch), int(limit_ns), ctypes.c_void_p(stream),
                                             ctypes.byref(b)))
    return b.value


def dmuon_momentum_norm_noalloc(grad: int, momentum: int, u_out: int, s_out: int, rows: int, cols: int,
                                grad_dtype="bf16", u_dtype="bf16", mu=0.95, nesterov=True, eps=1e-7, stream: int = 0):
    """Momentum + normalisation pass of one matrix with no workspace (see include/dmuon.h)."""
    _check(lib().dmuon_momentum_norm_noalloc(ctypes.c_void_p(grad), ctypes.c_void_p(momentum), ctypes.c_void_p(u_out),
                                             ctypes.c_void_p(s_out), int(rows), int(cols), DTYPE[grad_dtype],
                                             DTYPE[u_dtype], float(mu), int(bool(nesterov)), float(eps),
                                             ctypes.c_void_p(stream)))


def dmuon_assign_owners(shapes, n_ranks, ns_steps=5, costs=None):
    """Owner rank per matrix and the predicted load per rank (host only)."""
    n = len(shapes)
    sh = (Shape * max(n, 1))(*[Shape(int(r), int(c)) for r, c in shapes])
    cs = (ctypes.c_double * n)(*costs) if costs is not None else None
    own = (ctypes.c_int32 * max(n, 1))()
    load = (ctypes.c_double * max(n_ranks, 1))()
    _check(lib().dmuon_assign_owners(sh if n else None, n, ns_steps, cs, n_ranks, own, load))
    return list(own)[:n], list(load)[:n_ranks]


def dmuon_adamw_flat(param: int, grad: int, exp_avg: int, exp_avg_sq: int, n: int, param_dtype="bf16",
                     grad_dtype="bf16", lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1,
                     stream: int = 0):
    """One AdamW step over a flat buffer (see include/dmuon.h)."""
    _check(lib().dmuon_adamw_flat(ctypes.c_void_p(param), ctypes.c_void_p(grad), ctypes.c_void_p(exp_avg),
                                  ctypes.c_void_p(exp_avg_sq), int(n), DTYPE[param_dtype], DTYPE[grad_dtype],
                                  float(lr), float(beta1), float(beta2), float(eps), float(weight_decay), int(step),
                                  ctypes.c_void_p(stream)))


@dataclass
class Muon:
    """Convenience holder: a plan plus its torch-allocated workspace.

    ``params``, ``grads`` and ``momenta`` are lists of CUDA tensors (one per
    matrix, contiguous, 16-byte aligned). Only memory and the stream come
    from torch; the step itself is ``dmuon_step``.
    """

    plan: Plan
    workspace: object  # torch.Tensor (uint8, cuda)

    @classmethod
    def create(cls, shapes, *, ns_steps=5, coeffs=(3.4445, -4.7750, 2.0315), eps=1e-7, param="bf16",
               grad="bf16", compute="bf16", flags=0, device=None, stream=None):
        import torch
        plan = dmuon_plan(shapes, ns_steps, coeffs, eps, param, grad, compute, flags)
        nbytes = plan.workspace_bytes()
        ws = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device or "cuda")
        base = ws.data_ptr()
        aligned = (base + 1023) // 1024 * 1024
        s = stream if stream is not None else torch.cuda.current_stream()
        plan.bind(aligned, nbytes, s.cuda_stream)
        return cls(plan, ws)

    def step(self, params, grads, momenta, *, lr, mu=0.95, nesterov=True, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        self.plan.step([t.data_ptr() for t in params] if not isinstance(params[0], int) else params,
                       [t.data_ptr() for t in grads] if not isinstance(grads[0], int) else grads,
                       [t.data_ptr() for t in momenta] if not isinstance(momenta[0], int) else momenta,
                       lr, mu, nesterov, s.cuda_stream)
