"""TP mode emulated on one GPU vs the oracle's TP mode: P partitions (address t on
partition t mod P) and per-rank local buffers of remote rows; outputs of every rank
(local and remote rows, entry rows, CSR), every partition's state and every buffer's
state bit-exact after every step."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from synth.configs import small

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from oracle import COLD, FREE, OracleTP
    from serving_step_sparse_gb300 import ula
    from serving_step_sparse_gb300.cache import UlaTP
    from tests.gpu_harness import (compare_states, expand_id_rows, gpu_state_in_oracle_terms,
                                   unpack_bits)
    from tests.harness import ID_ROW_BYTES, alloc_rows, apply_events, initial_allocs


class _Geo:
    def __init__(self, S, H, B):
        self.gpu_slots, self.host_slots, self.ring_buckets = S, H, B


def _rows(w, base, n):
    G, L, W = w.n_groups, w.layers_per_group, w.row_bytes
    out = np.empty((G, n, L, W), dtype=np.uint8)
    for g in range(G):
        synth.content_range(w.seed, g, L, base, n, W, out=out[g])
    return out


def _buffer_state(st, slots, B):
    m = st["map"]
    where = np.where(m == ula.MAP_UNALLOCATED, -1, m.astype(np.int64))
    bits = np.stack([unpack_bits(st["class_bits"][c], slots) for c in range(B + 2)])
    which = bits.argmax(axis=0)
    cls = np.where(which < B, which, np.where(which == B, COLD, FREE)).astype(np.int32)
    return where, st["owner"], cls, st["cur"]


def run_tp(w, P, steps, buffer_slots=None, mode="bytes", sample_rows=None, seed=0):
    """mode "id": the oracle holds 8-byte id rows (exact: a row's bytes are a function of
    its address) and the gathered bytes are compared on sample_rows rows per output."""
    G, L, W, R = w.n_groups, w.layers_per_group, w.row_bytes, w.n_live
    E = w.entries_per_step
    S = -(-w.gpu_slots // P)
    H = -(-w.max_live_history // P) - S + E
    slots = buffer_slots or 2 * E
    tp = UlaTP(row_bytes=W, layers_per_group=[L] * G, parts=P, gpu_slots=S, host_slots=H,
               ring_buckets=w.ring_buckets, max_logical=w.max_logical, max_entries=E,
               buffer_slots=slots)
    orc = OracleTP(W if mode == "bytes" else ID_ROW_BYTES, [L] * G, P, S, H, w.ring_buckets,
                   w.max_logical, slots)
    rng = np.random.default_rng(seed)
    trace = synth.Trace(w)
    dev = tp.device

    def alloc(base, n):
        for off in range(0, n, 16384):  # staged in pieces
            m = min(16384, n - off)
            rows = _rows(w, base + off, m)
            t = torch.from_numpy(rows.reshape(-1)).pin_memory()
            assert tp.alloc(m, t) == base + off
            tp.sync()
            orows = rows.reshape(-1) if mode == "bytes" else alloc_rows(w, base + off, m, "id")
            assert orc.alloc(m, orows) == base + off
        return base

    def free(base, n):
        tp.free(base, n)
        orc.free(base, n)

    for base, n in initial_allocs(w, trace):
        alloc(base, n)
    lo = [tp.out_buffer(g, E) for g in range(G) for _ in range(P)]
    ro_ = [tp.out_buffer(g, E) for g in range(G) for _ in range(P)]
    mk = lambda n: [torch.empty(n, dtype=torch.int32, device=dev) for _ in range(P)]
    fetched = hits = remote = 0
    try:
        for t in range(steps):
            sel, ev = trace.step()
            sel_d = torch.from_numpy(np.ascontiguousarray(sel).view(np.int32)).to(dev)
            for g in range(G):
                louts, routs = lo[g * P:(g + 1) * P], ro_[g * P:(g + 1) * P]
                ler, lro, rer, rro = mk(E), mk(R + 1), mk(E), mk(R + 1)
                tp.step_group(g, sel_d[g], louts, routs, ler, lro, rer, rro)
                stats = tp.sync()
                res = orc.step_group(g, sel[g], out_cap=E)
                where = f"step {t} group {g}"
                for r in range(P):
                    for side, out, er, rq in (("local", louts, ler, lro), ("remote", routs, rer, rro)):
                        o = res[r][side]
                        U = int(o["req_off"][-1])
                        assert np.array_equal(rq[r].cpu().numpy(), o["req_off"]), f"{where} {side} {r}"
                        assert np.array_equal(er[r].cpu().numpy(), o["entry_row"]), f"{where} {side} {r}"
                        if mode == "bytes":
                            assert np.array_equal(out[r][:, :U].cpu().numpy(), o["out"][:, :U]), \
                                f"{where} {side} rows {r}"
                        else:
                            rows = rng.choice(U, min(U, sample_rows), replace=False) if U else np.zeros(0, int)
                            rt = torch.from_numpy(rows).to(dev)
                            for j in range(L):
                                got = out[r][j].index_select(0, rt).cpu().numpy()
                                exp = expand_id_rows(o["out"][j, rows], w.seed, g, j, W)
                                assert np.array_equal(got, exp), f"{where} {side} rows {r} layer {j}"
                    # partition r's state
                    go = gpu_state_in_oracle_terms(tp.parts[r].export(g), _Geo(S, H, w.ring_buckets))
                    compare_states(go, orc.partition(r).export(g), f"{where} partition {r}")
                    # rank r's buffer
                    gw, gown, gcls, gcur = _buffer_state(tp.buffers[r].export(g), slots,
                                                         w.ring_buckets)
                    ob = orc.buffer(r, g)
                    assert np.array_equal(gw, ob["where"]), f"{where} buffer {r} map"
                    assert np.array_equal(gown, ob["owner"]), f"{where} buffer {r} owners"
                    assert np.array_equal(gcls, ob["cls"]), f"{where} buffer {r} labels"
                    assert gcur == ob["cur"]
                    c = res[r]["remote"]["counters"]
                    fetched += c["misses"]
                    hits += c["hits"]
                    remote += c["uniq"]
            apply_events(alloc, free, ev)
        return fetched, hits, remote, stats
    finally:
        tp.close()


@pytest.mark.parametrize("name,P", [("tiny_1x4k", 2), ("batch8_32k", 2), ("batch8_32k", 4),
                                    ("longdoc", 4), ("low_overlap", 2)])
def test_tp_parity(name, P):
    from synth.configs import WORKLOADS
    w = WORKLOADS[name] if name == "tiny_1x4k" else small(name)
    w = w.replace(steps=min(w.steps, 16))
    fetched, hits, remote, stats = run_tp(w, P, w.steps)
    assert remote > 0 and hits > 0 and fetched > 0
    # fetched bytes are the buffers' fills
    assert sum(s["bytes_h2d"] for s in stats[P:]) == fetched * w.layers_per_group * w.row_bytes


def test_tp_full_size_sampled():
    """The long-document workload at full size with 4 partitions (oracle in id mode):
    states and entry rows exact, gathered bytes on sampled rows."""
    from synth.configs import WORKLOADS
    w = WORKLOADS["longdoc"]
    fetched, hits, remote, stats = run_tp(w, 4, 3, mode="id", sample_rows=2048)
    assert hits > 0 and fetched > 0


def test_tp_small_buffer_recycles_slots():
    w = small("batch8_32k").replace(steps=12)
    E = w.entries_per_step
    run_tp(w, 2, w.steps, buffer_slots=E)  # exactly one step's worth: evictions every step


def test_tp_validation():
    """Out-of-range partition counts, a zero-slot buffer and the unsupported option
    combinations are refused before anything is created."""
    L, W, S, H = 1, 16, 4, 4
    gp = [torch.empty(S * L * W, dtype=torch.uint8, device="cuda") for _ in range(9)]
    hp = [torch.empty(H * L * W, dtype=torch.uint8, pin_memory=True) for _ in range(9)]
    bp = [torch.empty(4 * L * W, dtype=torch.uint8, device="cuda") for _ in range(9)]
    ptrs = lambda xs, n: [x.data_ptr() for x in xs[:n]]
    for parts, slots, flags in ((0, 4, 0), (9, 4, 0), (2, 0, 0), (2, 4, ula.FLAG_EXACT_LRU),
                                (2, 4, ula.FLAG_LAYER_SIGNAL)):
        cfg = ula.make_config(W, [L], S, H, 2, 64, 8, flags)
        n = max(parts, 1)
        with pytest.raises(ula.UlaError) as ei:
            ula.ula_tp_create(cfg, parts, slots, ptrs(gp, n), ptrs(hp, n), ptrs(bp, n), None)
        assert ei.value.code == ula.ERR_INVALID_ARG
    cfg = ula.make_config(W, [L], S, H, 2, 64, 8, 0)
    tp = ula.ula_tp_create(cfg, 2, 4, ptrs(gp, 2), ptrs(hp, 2), ptrs(bp, 2), None)
    assert ula.ula_tp_context(tp, 0, 1) and ula.ula_tp_context(tp, 1, 1)
    assert ula.ula_tp_context(tp, 0, 2) == 0 and ula.ula_tp_context(tp, 2, 0) == 0
    with pytest.raises(ula.UlaError):  # beyond what was allocated
        ula.ula_tp_free(tp, 0, 1)
    ula.ula_tp_destroy(tp)
