"""TEST INFRASTRUCTURE: the CPU oracle of the KV residency path.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (``serving_step_sparse_gb300``)
never does; it has no CPU fallback.

The oracle is ``ula_oracle.cpp``: a plain single-threaded restatement of the
method on the UlaCache summary page (§2 "Unified logical addresses", §3
"PB-LRU"), with its own ordered-set containers.  This wrapper compiles it on
first use (g++, seconds) and marshals numpy arrays through ctypes.

Parity status of each part (pins live in ``tests/test_oracle_pins.py``):
  dedup / translate / gather -- pinned (closed form: gathered bytes equal the
      generator's row for the selected address; first-occurrence properties)
  never-both / slot ownership -- pinned (bijection invariant after every call)
  victim order -- pinned (brute-force round-granular LRU when no fold can
      happen; brute-force timestamp characterisation with folds; a hand-worked
      example)
  write-back host slots -- pinned (brute force from the exported state)
  timestamps (round of each slot's last access) -- pinned (brute force)
  exact-LRU mode (flag EXACT_LRU: timestamps + oldest-first victims) -- pinned
      (brute-force timestamp LRU on random tiny traces, with and without the
      overflow bypass)
  exact-LRU hit-rate companion (ExactLru) -- pinned through the exact-LRU mode
      (same hits on the same trace)
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, INVALID_ARG, CAPACITY, UNMAPPED, INTERNAL = 0, 1, 2, 3, 7
BYPASS = 1     # overflow bypass flag
EXACT_LRU = 2  # exact LRU in place of PB-LRU
FREE, COLD = -1, -2
TIER_UNALLOCATED, TIER_GPU, TIER_HOST = 0, 1, 2


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "ula_oracle.cpp")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-Wall", "-o", tmp, src],
                   check=True)
    os.replace(tmp, _SO)
    return _SO


def _configure(l):
    p, u32, i32 = C.c_void_p, C.c_uint32, C.c_int
    l.orc_create.argtypes = [u32, u32, p, u32, u32, u32, u32]
    l.orc_create.restype = p
    l.orc_create2.argtypes = [u32, u32, p, u32, u32, u32, u32, u32]
    l.orc_create2.restype = p
    l.orc_destroy.argtypes = [p]
    l.orc_alloc.argtypes = [p, u32, p, p]
    l.orc_alloc.restype = i32
    l.orc_free.argtypes = [p, u32, u32]
    l.orc_free.restype = i32
    l.orc_step_group.argtypes = [p, u32, p, u32, u32, u32, p, u32, p, p, p]
    l.orc_step_group.restype = i32
    l.orc_last_decisions.argtypes = [p, u32, p, p, p, p]
    l.orc_last_decisions.restype = u32
    l.orc_export.argtypes = [p, u32, p, p, p, p, p, p, p]
    l.orc_export_stamps.argtypes = [p, u32, p, p]
    l.orc_gpu_pool.argtypes = [p, u32]
    l.orc_gpu_pool.restype = p
    l.orc_host_pool.argtypes = [p, u32]
    l.orc_host_pool.restype = p
    l.orc_lru_create.argtypes = [u32, u32, u32]
    l.orc_lru_create.restype = p
    l.orc_lru_destroy.argtypes = [p]
    l.orc_lru_alloc.argtypes = [p, u32, p]
    l.orc_lru_alloc.restype = i32
    l.orc_lru_free.argtypes = [p, u32, u32]
    l.orc_lru_free.restype = i32
    l.orc_lru_step.argtypes = [p, u32, p, C.c_size_t, p]
    l.orc_lru_step.restype = i32
    l.orc_tp_create.argtypes = [u32, u32, p, u32, u32, u32, u32, u32, u32]
    l.orc_tp_create.restype = p
    l.orc_tp_destroy.argtypes = [p]
    l.orc_tp_alloc.argtypes = [p, u32, p, p]
    l.orc_tp_alloc.restype = i32
    l.orc_tp_free.argtypes = [p, u32, u32]
    l.orc_tp_free.restype = i32
    l.orc_tp_step_group.argtypes = [p, u32, p, u32, u32, u32, p, p, u32, p, p, p, p, p]
    l.orc_tp_step_group.restype = i32
    l.orc_tp_buffer.argtypes = [p, u32, u32, p, p, p, p, p]
    l.orc_tp_buffer.restype = u32
    l.orc_tp_partition.argtypes = [p, u32]
    l.orc_tp_partition.restype = p
    return l


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(C.CDLL(build()))
    return _lib


def load_variant(path: str):
    """Load another build of the oracle source (used by the mutation tests)."""
    return _configure(C.CDLL(path))


def _ptr(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags.c_contiguous
    return a.ctypes.data


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} -> status {code}")
        self.code = code


class Oracle:
    """Residency oracle (PB-LRU, or exact LRU): same calls as the library, semantically."""

    def __init__(self, row_bytes, layers_per_group, gpu_slots, host_slots, ring_buckets,
                 max_logical, _lib=None, bypass=False, exact_lru=False):
        self._l = _lib if _lib is not None else lib()
        self.row_bytes = int(row_bytes)
        self.layers = [int(x) for x in layers_per_group]
        self.G = len(self.layers)
        self.S, self.H, self.B = int(gpu_slots), int(host_slots), int(ring_buckets)
        self.max_logical = int(max_logical)
        L = np.array(self.layers, dtype=np.uint32)
        self.bypass = bool(bypass)
        self.exact_lru = bool(exact_lru)
        flags = (BYPASS if self.bypass else 0) | (EXACT_LRU if self.exact_lru else 0)
        if flags:
            self._h = self._l.orc_create2(self.row_bytes, self.G, _ptr(L), self.S, self.H,
                                          self.B, self.max_logical, flags)
        else:
            self._h = self._l.orc_create(self.row_bytes, self.G, _ptr(L), self.S, self.H,
                                         self.B, self.max_logical)
        if not self._h:
            raise ValueError("bad oracle configuration")

    def close(self):
        if self._h:
            self._l.orc_destroy(self._h)
            self._h = None

    __del__ = close

    def alloc(self, n: int, rows: np.ndarray | None) -> int:
        """rows: uint8 buffer holding, per group, [n][L_g][row_bytes]."""
        base = C.c_uint32(0)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.uint8)
            need = n * sum(self.layers) * self.row_bytes
            assert rows.size == need, (rows.size, need)
        rc = self._l.orc_alloc(self._h, n, _ptr(rows), C.byref(base))
        if rc:
            raise OracleError(rc, "alloc")
        return base.value

    def free(self, base: int, n: int):
        rc = self._l.orc_free(self._h, base, n)
        if rc:
            raise OracleError(rc, "free")

    def step_group(self, g: int, sel: np.ndarray, out_cap: int | None = None):
        """sel: uint32 [R][Q][k].  Returns dict(out [L][cap][W], entry_row, req_off, counters)."""
        sel = np.ascontiguousarray(sel, dtype=np.uint32)
        R, Q, K = sel.shape
        cap = int(out_cap if out_cap is not None else max(1, sel.size))
        out = np.zeros((self.layers[g], cap, self.row_bytes), dtype=np.uint8)
        entry_row = np.empty(sel.size, dtype=np.int32)
        req_off = np.empty(R + 1, dtype=np.int32)
        cnt = np.zeros(9, dtype=np.uint64)
        rc = self._l.orc_step_group(self._h, g, _ptr(sel), R, Q, K, _ptr(out), cap,
                                  _ptr(entry_row), _ptr(req_off), _ptr(cnt))
        if rc:
            raise OracleError(rc, f"step_group({g})")
        keys = ["uniq", "hits", "misses", "victims_free", "victims_cold", "victims_ring",
                "writebacks", "rows_gathered", "bypassed"]
        return {"out": out, "entry_row": entry_row, "req_off": req_off,
                "counters": {k: int(v) for k, v in zip(keys, cnt)}}

    def last_decisions(self, g: int):
        cap = self.S
        v = np.empty(cap, dtype=np.uint32)
        vc = np.empty(cap, dtype=np.int32)
        wb = np.empty(max(cap, 1), dtype=np.uint32)
        nwb = C.c_uint32(0)
        m = self._l.orc_last_decisions(self._h, g, _ptr(v), _ptr(vc), _ptr(wb), C.byref(nwb))
        return v[:m].copy(), vc[:m].copy(), wb[:nwb.value].copy()

    def export(self, g: int):
        tier = np.empty(self.max_logical, dtype=np.uint8)
        slot = np.empty(self.max_logical, dtype=np.uint32)
        cls = np.empty(self.S, dtype=np.int32)
        owner = np.empty(self.S, dtype=np.uint32)
        host_free = np.empty(max(self.H, 1), dtype=np.uint8)
        host_owner = np.empty(max(self.H, 1), dtype=np.uint32)
        cur = C.c_uint32(0)
        self._l.orc_export(self._h, g, _ptr(tier), _ptr(slot), _ptr(cls), _ptr(owner),
                         _ptr(host_free), _ptr(host_owner), C.byref(cur))
        return {"tier": tier, "slot": slot, "cls": cls, "owner": owner,
                "host_free": host_free[:self.H], "host_owner": host_owner[:self.H],
                "cur": cur.value}

    def stamps(self, g: int):
        """(timestamp per GPU slot: round of its last access, 0xFFFFFFFF if free; rounds so far)."""
        st = np.empty(self.S, dtype=np.uint32)
        r = C.c_uint32(0)
        self._l.orc_export_stamps(self._h, g, _ptr(st), C.byref(r))
        return st, r.value

    def gpu_pool(self, g: int) -> np.ndarray:
        n = self.S * self.layers[g] * self.row_bytes
        buf = (C.c_uint8 * n).from_address(self._l.orc_gpu_pool(self._h, g))
        return np.frombuffer(buf, dtype=np.uint8).reshape(self.S, self.layers[g], self.row_bytes)

    def host_pool(self, g: int) -> np.ndarray:
        n = self.H * self.layers[g] * self.row_bytes
        if n == 0:
            return np.zeros((0, self.layers[g], self.row_bytes), dtype=np.uint8)
        buf = (C.c_uint8 * n).from_address(self._l.orc_host_pool(self._h, g))
        return np.frombuffer(buf, dtype=np.uint8).reshape(self.H, self.layers[g], self.row_bytes)


class OracleTP:
    """TP mode emulated: P partitions (DP residency over t mod P) and, per rank and
    group, a local buffer of remote rows."""

    KEYS = ["uniq", "hits", "misses", "victims_free", "victims_cold", "victims_ring",
            "writebacks", "rows_gathered", "bypassed"]

    def __init__(self, row_bytes, layers_per_group, parts, gpu_slots, host_slots, ring_buckets,
                 max_logical, buffer_slots, _lib=None):
        self._l = _lib if _lib is not None else lib()
        self.row_bytes = int(row_bytes)
        self.layers = [int(x) for x in layers_per_group]
        self.G, self.P = len(self.layers), int(parts)
        self.S, self.H, self.B = int(gpu_slots), int(host_slots), int(ring_buckets)
        self.max_logical, self.slots = int(max_logical), int(buffer_slots)
        L = np.array(self.layers, dtype=np.uint32)
        self._h = self._l.orc_tp_create(self.row_bytes, self.G, _ptr(L), self.P, self.S, self.H,
                                        self.B, self.max_logical, self.slots)
        if not self._h:
            raise ValueError("bad TP oracle configuration")
        self._keep = L

    def close(self):
        if self._h:
            self._l.orc_tp_destroy(self._h)
            self._h = None

    __del__ = close

    def alloc(self, n: int, rows: np.ndarray | None) -> int:
        """rows: per group, [n][L_g][row_bytes] in global address order."""
        base = C.c_uint32(0)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.uint8)
        rc = self._l.orc_tp_alloc(self._h, n, _ptr(rows), C.byref(base))
        if rc:
            raise OracleError(rc, "tp alloc")
        return base.value

    def free(self, base: int, n: int):
        rc = self._l.orc_tp_free(self._h, base, n)
        if rc:
            raise OracleError(rc, "tp free")

    def step_group(self, g: int, sel: np.ndarray, out_cap: int | None = None):
        """Per rank r: res[r]["local"] (partition r's DP step on the entries it owns) and
        res[r]["remote"] (rank r's buffer on the entries it does not own), each a dict of
        out [L][cap][W], entry_row, req_off, counters."""
        sel = np.ascontiguousarray(sel, dtype=np.uint32)
        R, Q, K = sel.shape
        cap = int(out_cap if out_cap is not None else max(1, sel.size))
        L, P = self.layers[g], self.P
        mk = lambda: {"out": np.zeros((L, cap, self.row_bytes), dtype=np.uint8),
                      "entry_row": np.empty(sel.size, dtype=np.int32),
                      "req_off": np.empty(R + 1, dtype=np.int32)}
        loc, rem = [mk() for _ in range(P)], [mk() for _ in range(P)]
        arr = lambda xs, k: (C.c_void_p * P)(*[x[k].ctypes.data for x in xs])
        cnt = np.zeros((P, 2, 9), dtype=np.uint64)
        rc = self._l.orc_tp_step_group(self._h, g, _ptr(sel), R, Q, K, arr(loc, "out"),
                                       arr(rem, "out"), cap, arr(loc, "entry_row"),
                                       arr(loc, "req_off"), arr(rem, "entry_row"),
                                       arr(rem, "req_off"), _ptr(cnt))
        if rc:
            raise OracleError(rc, f"tp step_group({g})")
        res = []
        for r in range(P):
            loc[r]["counters"] = dict(zip(self.KEYS, map(int, cnt[r, 0])))
            rem[r]["counters"] = dict(zip(self.KEYS, map(int, cnt[r, 1])))
            res.append({"local": loc[r], "remote": rem[r]})
        return res

    def buffer(self, r: int, g: int):
        where = np.empty(self.max_logical, dtype=np.int64)
        owner = np.empty(self.slots, dtype=np.uint32)
        cls = np.empty(self.slots, dtype=np.int32)
        victims = np.empty(max(1, self.slots), dtype=np.uint32)
        cur = C.c_uint32(0)
        n = self._l.orc_tp_buffer(self._h, r, g, _ptr(where), _ptr(owner), _ptr(cls), C.byref(cur),
                                  _ptr(victims))
        return {"where": where, "owner": owner, "cls": cls, "cur": cur.value,
                "victims": victims[:n].copy()}

    def partition(self, p: int) -> "Oracle":
        """A non-owning view of partition p (its export and pools)."""
        o = _PartitionView.__new__(_PartitionView)
        o._l, o._h = self._l, self._l.orc_tp_partition(self._h, p)
        o.row_bytes, o.layers, o.G = self.row_bytes, self.layers, self.G
        o.S, o.H, o.B = self.S, self.H, self.B
        o.max_logical = (self.max_logical + self.P - 1) // self.P
        o.bypass = o.exact_lru = False
        o._owner = self  # keeps the TP oracle alive while the view is used
        return o


class _PartitionView(Oracle):
    """A partition of an OracleTP, seen as a DP oracle; it does not own the handle."""

    def close(self):
        self._h = None

    __del__ = close


class ExactLru:
    """Exact (round-granular) LRU companion; reports hit counts only."""

    def __init__(self, n_groups, gpu_slots, max_logical):
        self._h = lib().orc_lru_create(n_groups, gpu_slots, max_logical)
        self.acc = np.zeros(2, dtype=np.uint64)

    def close(self):
        if self._h:
            lib().orc_lru_destroy(self._h)
            self._h = None

    __del__ = close

    def alloc(self, n):
        base = C.c_uint32(0)
        rc = lib().orc_lru_alloc(self._h, n, C.byref(base))
        if rc:
            raise OracleError(rc, "lru alloc")
        return base.value

    def free(self, base, n):
        lib().orc_lru_free(self._h, base, n)

    def step_group(self, g, sel):
        sel = np.ascontiguousarray(sel, dtype=np.uint32)
        rc = lib().orc_lru_step(self._h, g, _ptr(sel), sel.size, _ptr(self.acc))
        if rc:
            raise OracleError(rc, "lru step")

    @property
    def hit_rate(self) -> float:
        return float(self.acc[1]) / max(1.0, float(self.acc[0]))
