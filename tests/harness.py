"""Test drivers: replay a synthetic workload through the oracle (and, for GPU
tests, through the library), plus the invariant checks both must satisfy.

Row modes:
  "bytes": 656-byte rows from the synth content generator (what the library moves)
  "id":    8-byte rows [addr u32][g<<16 | j u32]; exact because a row's content is a
           pure function of (group, layer, address), so the oracle can run the large
           workloads in id mode and the gathered ids are expanded to bytes for checks.
"""
from __future__ import annotations

import numpy as np

import synth
from oracle import COLD, FREE, TIER_GPU, TIER_HOST, TIER_UNALLOCATED, Oracle

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


def check_step_outputs(sel_g, res, g, w, mode):
    """Closed-form checks of one group-step's outputs (independent of the state)."""
    flat = sel_g.reshape(-1)
    entry_row, req_off = res["entry_row"], res["req_off"]
    U = int(req_off[-1])
    R = sel_g.shape[0]
    qk = sel_g.shape[1] * sel_g.shape[2]
    valid = flat != synth.PAD
    # dedup: distinct rows, ordered by first occurrence, every entry maps to its address
    assert (entry_row[~valid] == -1).all()
    rows = entry_row[valid]
    assert rows.min(initial=0) >= 0 and (rows < U).all()
    uniq = np.empty(U, dtype=np.uint32)
    uniq[rows] = flat[valid]
    assert len(np.unique(uniq)) == U
    first_entry = np.full(U, -1, dtype=np.int64)
    idx = np.nonzero(valid)[0]
    for e, r in zip(idx, rows):  # small cases only
        if first_entry[r] < 0:
            first_entry[r] = e
    assert (first_entry >= 0).all() and (np.diff(first_entry) > 0).all()
    # CSR by request: rows first seen in request r's entries are [req_off[r], req_off[r+1])
    for r in range(R):
        fe = first_entry[req_off[r]:req_off[r + 1]]
        assert ((fe >= r * qk) & (fe < (r + 1) * qk)).all()
    assert (np.diff(req_off) >= 0).all() and req_off[0] == 0
    # gather: out[j][u] is row j of uniq[u] (closed form from the generator)
    out = res["out"]
    for j in range(w.layers_per_group):
        got = out[j, :U]
        if mode == "bytes":
            exp = synth.content_list(w.seed, g, j, uniq, w.row_bytes)
        else:
            exp = np.empty((U, 2), dtype=np.uint32)
            exp[:, 0] = uniq
            exp[:, 1] = (g << 16) | j
            exp = exp.view(np.uint8).reshape(U, ID_ROW_BYTES)
        assert np.array_equal(got, exp), f"gathered rows differ (group {g}, layer {j})"
    return uniq


def check_invariants(st, S, H, live):
    """One tier per entry, slot ownership, class partition (oracle export format)."""
    tier, slot, cls, owner = st["tier"], st["slot"], st["cls"], st["owner"]
    host_free, host_owner = st["host_free"], st["host_owner"]
    live_arr = np.array(sorted(live), dtype=np.int64)
    alloc_mask = tier != TIER_UNALLOCATED
    assert alloc_mask.sum() == len(live_arr)
    assert alloc_mask[live_arr].all() if len(live_arr) else True
    gpu_addrs = np.nonzero(tier == TIER_GPU)[0]
    host_addrs = np.nonzero(tier == TIER_HOST)[0]
    # every live address has exactly one location, and the slot names it back
    assert len(np.unique(slot[gpu_addrs])) == len(gpu_addrs)
    assert len(np.unique(slot[host_addrs])) == len(host_addrs)
    assert (owner[slot[gpu_addrs]] == gpu_addrs).all()
    assert (host_owner[slot[host_addrs]] == host_addrs).all()
    occupied = owner != 0xFFFFFFFF
    assert occupied.sum() == len(gpu_addrs)
    # free class = unowned slots; classes partition the pool
    assert ((cls == FREE) == ~occupied).all()
    assert ((cls >= 0) | (cls == COLD) | (cls == FREE)).all()
    host_occ = host_owner != 0xFFFFFFFF
    assert host_occ.sum() == len(host_addrs)
    assert ((host_free == 1) == ~host_occ).all()
