"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle's tests.

Holds only random numbers and the workload recipe (row contents, per-step
top-k selections, request arrivals/appends); none of the residency method's
arithmetic.  The C source is ``synth.c``; this wrapper builds it on first use
(gcc, seconds) and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

from .configs import WORKLOADS, Workload, get_workload  # noqa: F401

PAD = 0xFFFFFFFF
_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into _build/libsynth.so (portable flags, OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall",
                    "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


class _Params(C.Structure):
    _fields_ = [("seed", C.c_uint64), ("n_groups", C.c_uint32), ("n_live", C.c_uint32),
                ("n_total", C.c_uint32), ("ctx_min", C.c_uint32), ("ctx_max", C.c_uint32),
                ("q", C.c_uint32), ("k", C.c_uint32), ("window", C.c_uint32),
                ("keep", C.c_double), ("fresh_zipf", C.c_uint32), ("zipf_s", C.c_double),
                ("append_max", C.c_uint32), ("append_cap", C.c_uint32),
                ("turnover_period", C.c_uint32), ("pad_prob", C.c_double)]


class _Events(C.Structure):
    _fields_ = [("free_base", C.c_uint32), ("free_n", C.c_uint32),
                ("append_base", C.c_uint32), ("append_n", C.c_uint32),
                ("join_base", C.c_uint32), ("join_n", C.c_uint32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            l = C.CDLL(build())
            p, u32, u64 = C.c_void_p, C.c_uint32, C.c_uint64
            l.synth_content_range.argtypes = [u64, u32, u32, u32, u32, u32, p]
            l.synth_content_list.argtypes = [u64, u32, u32, p, u32, u32, p]
            l.synth_trace_create.argtypes = [C.POINTER(_Params)]
            l.synth_trace_create.restype = p
            l.synth_trace_destroy.argtypes = [p]
            l.synth_trace_initial.argtypes = [p, p, p]
            l.synth_trace_initial.restype = u32
            l.synth_request_ctx.argtypes = [C.POINTER(_Params), u32]
            l.synth_request_ctx.restype = u32
            l.synth_trace_step.argtypes = [p, p, C.POINTER(_Events)]
            l.synth_trace_next_logical.argtypes = [p]
            l.synth_trace_next_logical.restype = u32
            _lib = l
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def content_range(seed: int, g: int, layers: int, addr0: int, n: int, row_bytes: int = 656,
                  out: np.ndarray | None = None) -> np.ndarray:
    """Rows [n][layers][row_bytes] (uint8) of group g for addresses addr0..addr0+n-1."""
    if out is None:
        out = np.empty((n, layers, row_bytes), dtype=np.uint8)
    assert out.dtype == np.uint8 and out.size >= n * layers * row_bytes
    if n:
        lib().synth_content_range(seed, g, layers, addr0, n, row_bytes, _ptr(out))
    return out


def content_list(seed: int, g: int, j: int, addrs: np.ndarray, row_bytes: int = 656) -> np.ndarray:
    """Rows [len(addrs)][row_bytes] of layer j of group g; PAD addresses give zero rows."""
    a = np.ascontiguousarray(addrs, dtype=np.uint32)
    out = np.empty((a.size, row_bytes), dtype=np.uint8)
    if a.size:
        lib().synth_content_list(seed, g, j, _ptr(a), a.size, row_bytes, _ptr(out))
    return out


def _params(w: Workload) -> _Params:
    return _Params(w.seed, w.n_groups, w.n_live, w.total_requests, w.ctx_min, w.ctx_max, w.q, w.k,
                   w.window, w.keep, 1 if w.fresh == "zipf" else 0, w.zipf_s, w.append_max,
                   w.append_cap, w.turnover_period, w.pad_prob)


def request_ctx(w: Workload, rid: int) -> int:
    p = _params(w)
    return int(lib().synth_request_ctx(C.byref(p), rid))


class Trace:
    """Stateful per-step selection generator for one workload.

    ``initial()`` gives the initial context lengths (live order); the library is
    expected to hand out logical ranges consecutively from 0 in that order.
    ``step()`` returns (sel [G][R][Q][k] uint32, events dict); the caller applies
    the events after the step's G group calls: free, then join, then appends.
    """

    def __init__(self, w: Workload):
        self.w = w
        self._p = _params(w)
        self._h = lib().synth_trace_create(C.byref(self._p))
        if not self._h:
            raise ValueError(f"bad workload parameters: {w}")

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.synth_trace_destroy(h)

    def initial(self):
        ctx = np.empty(self.w.n_live, dtype=np.uint32)
        base = np.empty(self.w.n_live, dtype=np.uint32)
        total = lib().synth_trace_initial(self._h, _ptr(ctx), _ptr(base))
        return ctx, base, int(total)

    def step(self):
        w = self.w
        sel = np.empty((w.n_groups, w.n_live, w.q, w.k), dtype=np.uint32)
        ev = _Events()
        lib().synth_trace_step(self._h, _ptr(sel), C.byref(ev))
        return sel, {f: int(getattr(ev, f)) for f, _ in _Events._fields_}

    def next_logical(self) -> int:
        return int(lib().synth_trace_next_logical(self._h))
