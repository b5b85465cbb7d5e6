"""UlaCache: one residency context plus the PyTorch plumbing around it.

PyTorch provides only device memory, pinned host memory and streams here; every
step of the path runs in the CUDA library through the C ABI (``ula``).
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import ula


def _thp_bytes() -> int:
    try:
        with open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size") as f:
            return int(f.read().strip())
    except (OSError, ValueError):
        return 2 << 20


def _huge_fraction(addr: int, nbytes: int) -> float | None:
    try:
        with open("/proc/self/smaps") as f:
            inside = False
            for line in f:
                head = line.split(None, 1)[0]
                if "-" in head and not head.endswith(":"):
                    lo, hi = (int(x, 16) for x in head.split("-"))
                    inside = lo <= addr < hi
                elif inside and head == "AnonHugePages:":
                    return min(1.0, int(line.split()[1]) * 1024 / max(1, nbytes))
    except (OSError, ValueError):
        pass
    return None


class PinnedHostBuffer:
    """Page-locked host memory for a host slot pool.

    An anonymous mapping aligned to the transparent-huge-page size, advised
    MADV_HUGEPAGE and registered with CUDA.  The kernels reach host slots at
    random over the host link; with base-size pages a pool of tens of GB needs
    more GPU address translations than stay cached, and random-slot bandwidth
    falls to about a third.  Huge pages keep the translations in reach.
    """

    def __init__(self, nbytes: int, huge: bool = True):
        import mmap
        self.nbytes = int(nbytes)
        align = _thp_bytes() if huge else mmap.PAGESIZE
        self._mm = mmap.mmap(-1, self.nbytes + align,
                             flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        if huge and hasattr(mmap, "MADV_HUGEPAGE"):
            self._mm.madvise(mmap.MADV_HUGEPAGE)
        whole = torch.frombuffer(self._mm, dtype=torch.uint8)
        off = (-whole.data_ptr()) % align
        self.tensor = whole[off:off + self.nbytes]
        del whole
        rt = torch.cuda.cudart()
        rc = rt.cudaHostRegister(self.tensor.data_ptr(), self.nbytes, 0)
        if getattr(rc, "value", rc) != 0:
            raise RuntimeError(f"cudaHostRegister failed: {rc}")
        self._registered = True

    def huge_fraction(self) -> float | None:
        """The fraction of the buffer backed by transparent huge pages (from the process's
        memory map), or None where that is not readable."""
        return _huge_fraction(self.tensor.data_ptr(), self.nbytes)

    def close(self):
        if getattr(self, "_registered", False):
            torch.cuda.cudart().cudaHostUnregister(self.tensor.data_ptr())
            self._registered = False
        self.tensor = None
        mm, self._mm = getattr(self, "_mm", None), None
        if mm is not None:
            try:
                mm.close()
            except BufferError:
                pass


def _u32(t: torch.Tensor) -> int:
    assert t.dtype in (torch.int32, torch.uint8) and t.is_contiguous()
    return t.data_ptr()


class UlaCache:
    """GPU slot pool + pinned host slot pool per layer group, one logical address space."""

    def __init__(self, *, row_bytes: int, layers_per_group, gpu_slots: int, host_slots: int,
                 ring_buckets: int, max_logical: int, max_entries: int, device="cuda",
                 stream: torch.cuda.Stream | None = None, huge_host_pages: bool = True,
                 bypass_overflow: bool = False, exact_lru: bool = False,
                 layer_signal: bool = False, gather_beside_move: bool = False):
        self.device = torch.device(device)
        self.W = int(row_bytes)
        self.layers = [int(x) for x in layers_per_group]
        self.G = len(self.layers)
        self.S, self.H, self.B = int(gpu_slots), int(host_slots), int(ring_buckets)
        self.max_logical, self.max_entries = int(max_logical), int(max_entries)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.gpu_pools = [torch.empty(self.S * L * self.W, dtype=torch.uint8, device=self.device)
                          for L in self.layers]
        self._host_bufs = ([PinnedHostBuffer(self.H * L * self.W, huge_host_pages)
                            for L in self.layers] if self.H else [])
        self.host_pools = [b.tensor for b in self._host_bufs] if self.H else None
        self.host_huge_fraction = [b.huge_fraction() for b in self._host_bufs] if self.H else []
        cfg = ula.make_config(self.W, self.layers, self.S, self.H, self.B, self.max_logical,
                              self.max_entries,
                              (ula.FLAG_BYPASS_OVERFLOW if bypass_overflow else 0)
                              | (ula.FLAG_EXACT_LRU if exact_lru else 0)
                              | (ula.FLAG_LAYER_SIGNAL if layer_signal else 0)
                              | (ula.FLAG_GATHER_BESIDE_MOVE if gather_beside_move else 0))
        with torch.cuda.device(self.device):
            self.ctx = ula.ula_create(cfg, [p.data_ptr() for p in self.gpu_pools],
                                      [p.data_ptr() for p in self.host_pools] if self.H else None,
                                      self.stream.cuda_stream)
        self.layout = ula.ula_debug_layout_get(self.ctx)

    # -- the five calls -------------------------------------------------------
    def alloc(self, n: int, rows: torch.Tensor) -> int:
        """rows: pinned host or device uint8 tensor holding, per group, [n][L_g][W]."""
        assert rows.dtype == torch.uint8 and rows.is_contiguous()
        assert rows.numel() == n * sum(self.layers) * self.W
        assert rows.is_cuda or rows.is_pinned()
        return ula.ula_alloc(self.ctx, n, rows.data_ptr())

    def free(self, base: int, n: int) -> None:
        ula.ula_free(self.ctx, base, n)

    def step_group(self, g: int, sel: torch.Tensor, out: torch.Tensor, entry_row: torch.Tensor,
                   req_off: torch.Tensor, layer_ready=None, stream: torch.cuda.Stream | None = None):
        """sel: device int32 view of uint32 [R][Q][k]; out: device uint8 [L][cap][W]."""
        R, Q, K = sel.shape
        cap = out.shape[1]
        s = stream if stream is not None else self.stream
        ev = None
        if layer_ready:
            for e in layer_ready:  # torch creates the CUDA event on first record
                if not e.cuda_event:
                    e.record(s)
            ev = [e.cuda_event for e in layer_ready]
        ula.ula_step_group(self.ctx, g, _u32(sel), R, Q, K, out.data_ptr(), cap,
                           _u32(entry_row), _u32(req_off), ev, s.cuda_stream)

    def layer_signal(self, g: int) -> tuple[int, int]:
        """(device address of group g's uint32 layer flags, round of its last step)."""
        return ula.ula_layer_signal(self.ctx, g)

    def sync(self) -> dict:
        return ula.ula_sync(self.ctx)

    def close(self):
        if getattr(self, "ctx", None):
            ula.ula_destroy(self.ctx)
            self.ctx = None
        self.host_pools = None
        for b in getattr(self, "_host_bufs", []):
            b.close()
        self._host_bufs = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- buffers --------------------------------------------------------------
    def out_buffer(self, g: int, cap: int) -> torch.Tensor:
        return torch.empty((self.layers[g], cap, self.W), dtype=torch.uint8, device=self.device)

    # -- diagnostics ----------------------------------------------------------
    def export(self, g: int) -> dict:
        lay = self.layout
        arrs = {
            "map": np.empty(self.max_logical, np.uint32),
            "owner": np.empty(self.S, np.uint32),
            "stamp": np.empty(self.S, np.uint32),
            "class_bits": np.empty((lay.n_classes, lay.n0), np.uint32),
            "class_sum1": np.empty((lay.n_classes, lay.n1), np.uint32),
            "class_sum2": np.empty((lay.n_classes, lay.n2), np.uint32),
            "host_free_bits": np.empty(max(lay.h0, 1), np.uint32),
            "host_free_sum1": np.empty(max(lay.h1, 1), np.uint32),
            "host_free_sum2": np.empty(max(lay.h2, 1), np.uint32),
            "uniq": np.empty(self.max_entries, np.uint32),
            "victims": np.empty(lay.decision_cap, np.uint32),
            "wb_host": np.empty(lay.decision_cap, np.uint32),
            "class_seg_count": np.empty((lay.n_classes, lay.n1), np.uint32),
            "host_seg_count": np.empty(max(lay.h1, 1), np.uint32),
            "row_slot": np.empty(self.max_entries, np.uint32),
        }
        st = ula.ula_debug_state()
        for k, a in arrs.items():
            setattr(st, k, a.ctypes.data)
        ula.ula_debug_export(self.ctx, g, st)
        for k in ("round", "cur", "free_gpu", "free_host", "U", "M", "hits", "victims_free",
                  "writebacks"):
            arrs[k] = int(getattr(st, k))
        return arrs

    def inject(self, code: int):
        ula.ula_debug_inject(self.ctx, code)


class _ContextView(UlaCache):
    """A context owned by a UlaTP, with UlaCache's diagnostics (export); not owned."""

    def __init__(self, ctx: int, gpu_slots: int, host_slots: int, max_logical: int,
                 max_entries: int, layers, row_bytes: int, ring_buckets: int, device):
        self.ctx = ctx
        self.S, self.H, self.B = gpu_slots, host_slots, ring_buckets
        self.max_logical, self.max_entries = max_logical, max_entries
        self.layers, self.W, self.G = list(layers), row_bytes, len(layers)
        self.device = device
        self._host_bufs = []
        self.layout = ula.ula_debug_layout_get(ctx)

    def close(self):
        self.ctx = None


class UlaTP:
    """TP mode emulated on one GPU: P partitions (address t on partition t mod P), each a
    DP residency with its own GPU and pinned host pools, and per rank a local buffer of
    remote rows (buffer_slots slots per group) filled from the owners' GPU pools."""

    def __init__(self, *, row_bytes: int, layers_per_group, parts: int, gpu_slots: int,
                 host_slots: int, ring_buckets: int, max_logical: int, max_entries: int,
                 buffer_slots: int, device="cuda", stream: torch.cuda.Stream | None = None,
                 huge_host_pages: bool = True):
        self.device = torch.device(device)
        self.W, self.layers, self.P = int(row_bytes), [int(x) for x in layers_per_group], int(parts)
        self.G = len(self.layers)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        P, S, H = self.P, int(gpu_slots), int(host_slots)
        self.gpu_pools = [torch.empty(S * L * self.W, dtype=torch.uint8, device=self.device)
                          for _ in range(P) for L in self.layers]
        self._host_bufs = ([PinnedHostBuffer(H * L * self.W, huge_host_pages)
                            for _ in range(P) for L in self.layers] if H else [])
        self.buffer_pools = [torch.empty(int(buffer_slots) * L * self.W, dtype=torch.uint8,
                                         device=self.device)
                             for _ in range(P) for L in self.layers]
        cfg = ula.make_config(self.W, self.layers, S, H, int(ring_buckets), int(max_logical),
                              int(max_entries), 0)
        with torch.cuda.device(self.device):
            self.tp = ula.ula_tp_create(cfg, P, int(buffer_slots),
                                        [t.data_ptr() for t in self.gpu_pools],
                                        [b.tensor.data_ptr() for b in self._host_bufs] if H else None,
                                        [t.data_ptr() for t in self.buffer_pools],
                                        self.stream.cuda_stream)
        local_max = (int(max_logical) + P - 1) // P
        self.parts = [_ContextView(ula.ula_tp_context(self.tp, 0, p), S, H, local_max,
                                   int(max_entries), self.layers, self.W, int(ring_buckets),
                                   self.device) for p in range(P)]
        self.buffers = [_ContextView(ula.ula_tp_context(self.tp, 1, r), int(buffer_slots), 0,
                                     int(max_logical), int(max_entries), self.layers, self.W,
                                     int(ring_buckets), self.device) for r in range(P)]

    def alloc(self, n: int, rows: torch.Tensor) -> int:
        """rows: pinned host or device uint8, per group [n][L_g][W] in global order."""
        return ula.ula_tp_alloc(self.tp, n, rows.data_ptr())

    def free(self, base: int, n: int):
        ula.ula_tp_free(self.tp, base, n)

    def step_group(self, g: int, sel: torch.Tensor, local_out, remote_out, local_entry_row,
                   local_req_off, remote_entry_row, remote_req_off):
        """sel: device int32 view of uint32 [R][Q][k]; the rest: lists of P device tensors."""
        R, Q, K = sel.shape
        cap = local_out[0].shape[1]
        ula.ula_tp_step_group(self.tp, g, sel.data_ptr(), R, Q, K,
                              [t.data_ptr() for t in local_out], [t.data_ptr() for t in remote_out],
                              cap, [t.data_ptr() for t in local_entry_row],
                              [t.data_ptr() for t in local_req_off],
                              [t.data_ptr() for t in remote_entry_row],
                              [t.data_ptr() for t in remote_req_off], self.stream.cuda_stream)

    def sync(self) -> list:
        """[2P] counter dicts: partitions, then the ranks' buffers."""
        return ula.ula_tp_sync(self.tp, self.P)

    def out_buffer(self, g: int, cap: int) -> torch.Tensor:
        return torch.empty((self.layers[g], cap, self.W), dtype=torch.uint8, device=self.device)

    def close(self):
        if getattr(self, "tp", None):
            ula.ula_tp_destroy(self.tp)
            self.tp = None
        for b in getattr(self, "_host_bufs", []):
            b.close()
        self._host_bufs = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
