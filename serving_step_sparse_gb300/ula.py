"""Thin Python binding of the C ABI in include/ula.h (ctypes; marshalling only).

Every step of the residency path runs in the CUDA library
``_build/libula.so``; this module only converts arguments.  There is no CPU
fallback: importing it without the built library raises ImportError.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libula.so")

MAX_GROUPS = 64
MAX_BUCKETS = 64
ADDR_PAD = 0xFFFFFFFF
FLAG_BYPASS_OVERFLOW = 1
FLAG_EXACT_LRU = 2
FLAG_LAYER_SIGNAL = 4
FLAG_GATHER_BESIDE_MOVE = 8
MAP_UNALLOCATED = 0xFFFFFFFF
MAP_HOST = 0x80000000
STAMP_FREE = 0xFFFFFFFF

OK = 0
ERR_INVALID_ARG = 1
ERR_CAPACITY = 2
ERR_UNMAPPED = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
DEBUG_STALL_SCAN_BARRIER = 0x100  # ula_debug_inject: the next exact-LRU scan waits out its barrier bound
ERR_POISONED = 6
ERR_INTERNAL = 7

PHASES = ["dedup", "rotate", "mark", "select", "move", "gather", "alloc", "free", "stage"]
NOALLOC_MAX_ENTRIES = 65536


class ula_config(C.Structure):
    _fields_ = [("row_bytes", C.c_uint32), ("n_groups", C.c_uint32),
                ("layers_per_group", C.c_uint32 * MAX_GROUPS), ("gpu_slots", C.c_uint32),
                ("host_slots", C.c_uint32), ("ring_buckets", C.c_uint32),
                ("max_logical", C.c_uint32), ("max_entries", C.c_uint32), ("flags", C.c_uint32)]


class ula_stats(C.Structure):
    _fields_ = [(n, C.c_uint64) for n in (
        "steps", "entries", "uniq", "hits", "misses", "victims_free", "victims_cold",
        "victims_ring", "writebacks", "rows_gathered", "bytes_h2d", "bytes_d2h", "bypassed")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class ula_debug_layout(C.Structure):
    _fields_ = [(n, C.c_uint32) for n in ("n0", "n1", "n2", "h0", "h1", "h2", "n_classes",
                                          "decision_cap")]


class ula_debug_state(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "map", "owner", "stamp", "class_bits", "class_sum1", "class_sum2", "host_free_bits",
        "host_free_sum1", "host_free_sum2", "uniq", "victims", "wb_host", "class_seg_count",
        "host_seg_count", "row_slot")] + \
        [(n, C.c_uint32) for n in ("round", "cur", "free_gpu", "free_host", "U", "M", "hits",
                                    "victims_free", "writebacks")]


class ula_profile(C.Structure):
    _fields_ = [("kernels", C.c_uint64 * len(PHASES)), ("timed", C.c_uint64 * len(PHASES)),
                ("ms", C.c_double * len(PHASES))]

    def as_dict(self):
        return {p: {"kernels": int(self.kernels[i]), "timed": int(self.timed[i]),
                    "ms": float(self.ms[i])} for i, p in enumerate(PHASES)}


class ula_span(C.Structure):
    _fields_ = [("phase", C.c_uint32), ("group", C.c_uint32), ("start_ns", C.c_uint64),
                ("end_ns", C.c_uint64)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library not built: {LIB_PATH} (run __graft_entry__.build())")
    lib = C.CDLL(LIB_PATH)
    p, u32, i32 = C.c_void_p, C.c_uint32, C.c_int
    lib.ula_create.argtypes = [C.POINTER(ula_config), p, p, p, C.POINTER(p)]
    lib.ula_create.restype = i32
    lib.ula_alloc.argtypes = [p, u32, p, C.POINTER(u32)]
    lib.ula_alloc.restype = i32
    lib.ula_free.argtypes = [p, u32, u32]
    lib.ula_free.restype = i32
    lib.ula_step_group.argtypes = [p, u32, p, u32, u32, u32, p, u32, p, p, p, p]
    lib.ula_step_group.restype = i32
    lib.ula_sync.argtypes = [p, C.POINTER(ula_stats)]
    lib.ula_sync.restype = i32
    lib.ula_destroy.argtypes = [p]
    lib.ula_destroy.restype = None
    lib.ula_error_string.argtypes = [i32]
    lib.ula_error_string.restype = C.c_char_p
    lib.ula_debug_layout_get.argtypes = [p, C.POINTER(ula_debug_layout)]
    lib.ula_debug_layout_get.restype = i32
    lib.ula_debug_export.argtypes = [p, u32, C.POINTER(ula_debug_state)]
    lib.ula_debug_export.restype = i32
    lib.ula_debug_inject.argtypes = [p, i32]
    lib.ula_debug_inject.restype = i32
    lib.ula_profile_enable.argtypes = [p, i32]
    lib.ula_profile_enable.restype = i32
    lib.ula_profile_read.argtypes = [p, C.POINTER(ula_profile), i32]
    lib.ula_profile_read.restype = i32
    lib.ula_profile_spans.argtypes = [p, i32]
    lib.ula_profile_spans.restype = i32
    lib.ula_profile_spans_read.argtypes = [p, p, u32, C.POINTER(u32)]
    lib.ula_profile_spans_read.restype = i32
    lib.ula_debug_regather.argtypes = [p, u32, u32, u32, p, u32, u32, p]
    lib.ula_debug_regather.restype = i32
    lib.ula_dedup_noalloc.argtypes = [p, u32, p, p, p, p]
    lib.ula_dedup_noalloc.restype = i32
    lib.ula_layer_signal.argtypes = [p, u32, C.POINTER(p), C.POINTER(u32)]
    lib.ula_layer_signal.restype = i32
    lib.ula_debug_layer_times.argtypes = [p, u32, p]
    lib.ula_debug_layer_times.restype = i32
    lib.ula_debug_consume.argtypes = [p, u32, u32, u32, p, u32, u32, p, p]
    lib.ula_debug_consume.restype = i32
    lib.ula_tp_create.argtypes = [C.POINTER(ula_config), u32, u32, p, p, p, p, C.POINTER(p)]
    lib.ula_tp_create.restype = i32
    lib.ula_tp_alloc.argtypes = [p, u32, p, C.POINTER(u32)]
    lib.ula_tp_alloc.restype = i32
    lib.ula_tp_free.argtypes = [p, u32, u32]
    lib.ula_tp_free.restype = i32
    lib.ula_tp_step_group.argtypes = [p, u32, p, u32, u32, u32, p, p, u32, p, p, p, p, p]
    lib.ula_tp_step_group.restype = i32
    lib.ula_tp_sync.argtypes = [p, p]
    lib.ula_tp_sync.restype = i32
    lib.ula_tp_context.argtypes = [p, i32, u32]
    lib.ula_tp_context.restype = p
    lib.ula_tp_destroy.argtypes = [p]
    lib.ula_tp_destroy.restype = i32
    return lib


lib = _load()


class UlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = lib.ula_error_string(code).decode()
        super().__init__(f"{what}: {msg} (code {code})")
        self.code = code


def _check(rc: int, what: str):
    if rc != OK:
        raise UlaError(rc, what)


def _ptr_array(ptrs):
    arr = (C.c_void_p * len(ptrs))()
    for i, x in enumerate(ptrs):
        arr[i] = x
    return arr


def make_config(row_bytes, layers_per_group, gpu_slots, host_slots, ring_buckets, max_logical,
                max_entries, flags=0) -> ula_config:
    cfg = ula_config()
    cfg.row_bytes = row_bytes
    cfg.n_groups = len(layers_per_group)
    for i, l in enumerate(layers_per_group):
        cfg.layers_per_group[i] = l
    cfg.gpu_slots, cfg.host_slots, cfg.ring_buckets = gpu_slots, host_slots, ring_buckets
    cfg.max_logical, cfg.max_entries, cfg.flags = max_logical, max_entries, flags
    return cfg


def ula_create(cfg: ula_config, gpu_pools, host_pools, stream: int | None) -> int:
    """gpu_pools/host_pools: lists of integer addresses; stream: cudaStream_t as int."""
    out = C.c_void_p()
    hp = _ptr_array(host_pools) if host_pools is not None else None
    _check(lib.ula_create(C.byref(cfg), _ptr_array(gpu_pools), hp, stream, C.byref(out)),
           "ula_create")
    return out.value


def ula_alloc(ctx: int, n: int, rows: int) -> int:
    base = C.c_uint32()
    _check(lib.ula_alloc(ctx, n, rows, C.byref(base)), "ula_alloc")
    return base.value


def ula_free(ctx: int, base: int, n: int) -> None:
    _check(lib.ula_free(ctx, base, n), "ula_free")


def ula_step_group(ctx: int, group: int, d_sel: int, n_req: int, q: int, k: int, d_out: int,
                   out_cap_rows: int, d_entry_row: int, d_req_off: int, layer_ready, stream) -> None:
    ev = _ptr_array(layer_ready) if layer_ready else None
    _check(lib.ula_step_group(ctx, group, d_sel, n_req, q, k, d_out, out_cap_rows, d_entry_row,
                              d_req_off, ev, stream), "ula_step_group")


def ula_sync(ctx: int) -> dict:
    st = ula_stats()
    _check(lib.ula_sync(ctx, C.byref(st)), "ula_sync")
    return st.as_dict()


def ula_sync_rc(ctx: int) -> int:
    """ula_sync returning the status code instead of raising."""
    return lib.ula_sync(ctx, None)


def ula_destroy(ctx: int) -> None:
    lib.ula_destroy(ctx)


def ula_debug_layout_get(ctx: int) -> ula_debug_layout:
    lay = ula_debug_layout()
    _check(lib.ula_debug_layout_get(ctx, C.byref(lay)), "ula_debug_layout_get")
    return lay


def ula_debug_export(ctx: int, group: int, st: ula_debug_state) -> ula_debug_state:
    _check(lib.ula_debug_export(ctx, group, C.byref(st)), "ula_debug_export")
    return st


def ula_layer_signal(ctx: int, group: int) -> tuple[int, int]:
    """(device address of the group's layer flags, round of its last issued step)."""
    ptr, rnd = C.c_void_p(), C.c_uint32()
    _check(lib.ula_layer_signal(ctx, group, C.byref(ptr), C.byref(rnd)), "ula_layer_signal")
    return ptr.value or 0, rnd.value


def ula_debug_layer_times(ctx: int, group: int, layers: int):
    """[L + 1] globaltimer ns: when each layer's flag was set, then the step's start."""
    import numpy as np
    ns = np.zeros(layers + 1, dtype=np.uint64)
    _check(lib.ula_debug_layer_times(ctx, group, ns.ctypes.data), "ula_debug_layer_times")
    return ns


def ula_debug_consume(ctx: int, group: int, layer: int, round_: int, d_out: int,
                      out_cap_rows: int, n_rows: int, d_result: int, stream) -> None:
    _check(lib.ula_debug_consume(ctx, group, layer, round_, d_out, out_cap_rows, n_rows,
                                 d_result, stream), "ula_debug_consume")


def ula_tp_create(cfg: ula_config, parts: int, buffer_slots: int, gpu_pools, host_pools,
                  buffer_pools, stream) -> int:
    out = C.c_void_p()
    hp = _ptr_array(host_pools) if host_pools else None
    _check(lib.ula_tp_create(C.byref(cfg), parts, buffer_slots, _ptr_array(gpu_pools), hp,
                             _ptr_array(buffer_pools), stream, C.byref(out)), "ula_tp_create")
    return out.value


def ula_tp_alloc(tp: int, n: int, rows: int) -> int:
    base = C.c_uint32()
    _check(lib.ula_tp_alloc(tp, n, rows, C.byref(base)), "ula_tp_alloc")
    return base.value


def ula_tp_free(tp: int, base: int, n: int) -> None:
    _check(lib.ula_tp_free(tp, base, n), "ula_tp_free")


def ula_tp_step_group(tp: int, group: int, d_sel: int, n_req: int, q: int, k: int, local_out,
                      remote_out, out_cap_rows: int, local_entry_row, local_req_off,
                      remote_entry_row, remote_req_off, stream) -> None:
    _check(lib.ula_tp_step_group(tp, group, d_sel, n_req, q, k, _ptr_array(local_out),
                                 _ptr_array(remote_out), out_cap_rows,
                                 _ptr_array(local_entry_row), _ptr_array(local_req_off),
                                 _ptr_array(remote_entry_row), _ptr_array(remote_req_off),
                                 stream), "ula_tp_step_group")


def ula_tp_sync(tp: int, parts: int) -> list:
    st = (ula_stats * (2 * parts))()
    _check(lib.ula_tp_sync(tp, C.cast(st, C.c_void_p)), "ula_tp_sync")
    return [s.as_dict() for s in st]


def ula_tp_context(tp: int, kind: int, index: int) -> int:
    return lib.ula_tp_context(tp, kind, index) or 0


def ula_tp_destroy(tp: int) -> None:
    lib.ula_tp_destroy(tp)


def ula_debug_inject(ctx: int, code: int) -> None:
    _check(lib.ula_debug_inject(ctx, code), "ula_debug_inject")


def ula_debug_regather(ctx: int, group: int, layer: int, d_out: int, out_cap_rows: int,
                       stream, blocks_per_sm: int = 0, n_layers: int = 1) -> None:
    _check(lib.ula_debug_regather(ctx, group, layer, n_layers, d_out, out_cap_rows,
                                  blocks_per_sm, stream), "ula_debug_regather")


def ula_profile_enable(ctx: int, on: bool) -> None:
    _check(lib.ula_profile_enable(ctx, 1 if on else 0), "ula_profile_enable")


def ula_profile_read(ctx: int, reset: bool = False) -> dict:
    pr = ula_profile()
    _check(lib.ula_profile_read(ctx, C.byref(pr), 1 if reset else 0), "ula_profile_read")
    return pr.as_dict()


def ula_profile_spans(ctx: int, on: bool) -> None:
    _check(lib.ula_profile_spans(ctx, 1 if on else 0), "ula_profile_spans")


def ula_profile_spans_read(ctx: int, cap: int = 1 << 16) -> list:
    """The recorded copy-kernel launch spans: [(phase name, group, start_ns, end_ns)]."""
    buf = (ula_span * cap)()
    n = C.c_uint32()
    _check(lib.ula_profile_spans_read(ctx, buf, cap, C.byref(n)), "ula_profile_spans_read")
    return [(PHASES[buf[i].phase], int(buf[i].group), int(buf[i].start_ns), int(buf[i].end_ns))
            for i in range(min(n.value, cap))]


def ula_dedup_noalloc(d_sel: int, n: int, d_uniq: int, d_entry_row: int, d_n_uniq: int,
                      stream) -> None:
    """First-occurrence dedup without a context and without allocating (fixed scratch)."""
    _check(lib.ula_dedup_noalloc(d_sel, n, d_uniq, d_entry_row, d_n_uniq, stream),
           "ula_dedup_noalloc")
