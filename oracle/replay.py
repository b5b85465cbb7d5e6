"""TEST INFRASTRUCTURE: replay of a synthetic workload through the oracle.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
use this module (the product path never does).  It holds no arithmetic of the
method: it feeds the seeded trace of ``synth`` (selections, joins, finishes,
appended tokens) into the oracle in the order the trace assigns logical ranges.

Row modes:
  "bytes": 656-byte rows from the synth content generator (what the library moves)
  "id":    8-byte rows [addr u32][g<<16 | j u32]; exact because a row's content is a
           pure function of (group, layer, address), so the oracle can run the large
           workloads in id mode and the gathered ids are expanded to bytes for checks.
"""
from __future__ import annotations

import numpy as np

import synth
from oracle import Oracle

ID_ROW_BYTES = 8


def id_rows(g: int, layers: int, addr0: int, n: int) -> np.ndarray:
    r = np.empty((n, layers, 2), dtype=np.uint32)
    r[:, :, 0] = (addr0 + np.arange(n, dtype=np.uint64)).astype(np.uint32)[:, None]
    r[:, :, 1] = (np.uint32(g) << np.uint32(16)) | np.arange(layers, dtype=np.uint32)[None, :]
    return r.view(np.uint8).reshape(n, layers, ID_ROW_BYTES)


def alloc_rows(w, addr0: int, n: int, mode: str) -> np.ndarray:
    """Flat uint8 buffer: for each group, [n][L_g][row_bytes] (groups concatenated)."""
    L = w.layers_per_group
    parts = []
    for g in range(w.n_groups):
        if mode == "bytes":
            parts.append(synth.content_range(w.seed, g, L, addr0, n, w.row_bytes).reshape(-1))
        else:
            parts.append(id_rows(g, L, addr0, n).reshape(-1))
    return np.concatenate(parts) if parts else np.zeros(0, np.uint8)


def make_oracle(w, mode: str = "bytes") -> Oracle:
    W = w.row_bytes if mode == "bytes" else ID_ROW_BYTES
    return Oracle(W, [w.layers_per_group] * w.n_groups, w.gpu_slots, w.host_slots,
                  w.ring_buckets, w.max_logical, bypass=w.bypass, exact_lru=w.exact_lru)


def initial_allocs(w, trace):
    """(base, n) of the initial contexts in live order (consecutive from 0)."""
    ctx, base, total = trace.initial()
    return [(int(b), int(c)) for b, c in zip(base, ctx)]


def apply_events(dev_alloc, dev_free, ev):
    """Apply a step's events in the order the generator assigned logical ranges."""
    if ev["free_n"]:
        dev_free(ev["free_base"], ev["free_n"])
    if ev["join_n"]:
        got = dev_alloc(ev["join_base"], ev["join_n"])
        assert got == ev["join_base"], (got, ev)
    if ev["append_n"]:
        got = dev_alloc(ev["append_base"], ev["append_n"])
        assert got == ev["append_base"], (got, ev)


class OracleRun:
    """A workload replayed on the oracle, step by step."""

    def __init__(self, w, mode: str = "bytes"):
        self.w, self.mode = w, mode
        self.o = make_oracle(w, mode)
        self.trace = synth.Trace(w)
        self.live = set()
        for base, n in initial_allocs(w, self.trace):
            self.alloc(base, n)

    def alloc(self, expect_base, n):
        got = self.o.alloc(n, alloc_rows(self.w, expect_base, n, self.mode))
        assert got == expect_base, (got, expect_base)
        self.live.update(range(got, got + n))
        return got

    def free(self, base, n):
        self.o.free(base, n)
        self.live.difference_update(range(base, base + n))

    def step(self):
        """One decode step: every group once, then the step's events."""
        sel, ev = self.trace.step()
        res = [self.o.step_group(g, sel[g]) for g in range(self.w.n_groups)]
        apply_events(self.alloc, self.free, ev)
        return sel, ev, res
