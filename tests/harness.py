"""Test checks: the invariants and closed forms that every replay (oracle or
library) must satisfy.  The replay drivers themselves are in ``oracle.replay``
and are re-exported here for the tests.
"""
from __future__ import annotations

import numpy as np

import synth
from oracle import COLD, FREE, TIER_GPU, TIER_HOST, TIER_UNALLOCATED
from oracle.replay import (ID_ROW_BYTES, OracleRun, alloc_rows, apply_events,  # noqa: F401
                           id_rows, initial_allocs, make_oracle)


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
