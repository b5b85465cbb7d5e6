"""The GPU path against the oracle over whole traces at full size.

Each workload's whole trace (512 or 256 decode steps) runs in the benchmark's launch
configuration (every group's call on its own caller stream).  After every step and for
every group: the CSR offsets equal the oracle's, the entry rows are equal (digest), and
the gathered rows equal the bytes of the oracle's unique addresses -- every row of every
layer on every 32nd step, 4,096 sampled rows per layer otherwise.  Every 16th step (and
the last): the full state -- map tier and slot of every address, class and owner and
timestamp of every GPU slot, host-free set and host-slot owners, the step's victims and
write-back slots -- equals the oracle's (digests), and the library's own summaries,
segment counts and stamps are consistent.  The oracle (id mode) runs in one spawned
process per group, concurrently with the GPU replay.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from synth.configs import WORKLOADS
from tests.full_trace import OracleWorkers, digest, state_digests

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from tests.gpu_harness import GpuReplay, check_gpu_internal, gpu_state_in_oracle_terms

from tests.harness import apply_events


def replay_full_trace(name, overrides=None, state_every=16, out_every=32, sample_rows=4096):
    w = WORKLOADS[name].replace(**overrides) if overrides else WORKLOADS[name]
    steps = w.steps
    G, L, W = w.n_groups, w.layers_per_group, w.row_bytes
    workers = OracleWorkers(name, overrides or {}, G, steps, state_every)
    gpu = None
    rng = np.random.default_rng(1234)
    counts = {"steps": 0, "rows_full": 0, "rows_sampled": 0, "states": 0}
    try:
        gpu = GpuReplay(w, group_streams=True)
        dev = gpu.cache.device
        for g in range(G):
            workers.recv(g, "ready")
        for t in range(steps):
            sel, ev = gpu.trace.step()
            gpu.run_groups(sel)
            for g in range(G):
                msg = workers.recv(g, "step")
                where = f"{name} step {t} group {g}"
                assert msg["t"] == t, where
                res = gpu.results(g, full_out=False)
                assert np.array_equal(res["req_off"], msg["req_off"]), f"{where}: req_off"
                assert digest(res["entry_row"]) == msg["entry_row"], f"{where}: entry rows"
                U, uniq = msg["U"], msg["uniq"]
                if t % out_every == 0:  # every gathered byte of every layer
                    for j in range(L):
                        exp = synth.content_list(w.seed, g, j, uniq, W)
                        got = gpu.outs[g][j][:U]
                        assert torch.equal(got, torch.from_numpy(exp).to(dev)), \
                            f"{where}: gathered bytes layer {j}"
                    counts["rows_full"] += U * L
                elif U:
                    pos = np.sort(rng.choice(U, min(U, sample_rows), replace=False))
                    pos_t = torch.from_numpy(pos).to(dev)
                    for j in range(L):
                        exp = synth.content_list(w.seed, g, j, uniq[pos], W)
                        got = gpu.outs[g][j].index_select(0, pos_t).cpu().numpy()
                        assert np.array_equal(got, exp), f"{where}: sampled rows layer {j}"
                    counts["rows_sampled"] += len(pos) * L
                if "state" in msg:
                    st = gpu.cache.export(g)
                    check_gpu_internal(st, w)
                    go = gpu_state_in_oracle_terms(st, w)
                    mine = state_digests(go, (st["victims"][:st["M"]],
                                              st["wb_host"][:st["writebacks"]]))
                    theirs = msg["state"]
                    diff = [k for k in theirs if mine.get(k) != theirs[k]]
                    assert not diff, f"{where}: state differs in {diff}"
                    counts["states"] += 1
            apply_events(gpu.alloc, gpu.free, ev)
            counts["steps"] += 1
        for g in range(G):
            workers.recv(g, "done")
        return gpu.cache.sync(), counts
    finally:
        workers.close()
        if gpu is not None:
            gpu.close()


@pytest.mark.parametrize("name", ["longdoc", "low_evict", "low_overlap", "low_overlap_256"])
def test_full_trace_bit_exact(name):
    w = WORKLOADS[name]
    stats, counts = replay_full_trace(name)
    assert counts["steps"] == w.steps and stats["steps"] == w.steps * w.n_groups
    assert counts["states"] == w.n_groups * (w.steps // 16 + (w.steps % 16 != 0))
    assert counts["rows_full"] > 0 and counts["rows_sampled"] > 0
    if w.bypass:
        assert stats["bypassed"] > 0
