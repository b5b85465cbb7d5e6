"""GPU path vs the CPU oracle: bit-exact on every map entry, class label,
eviction decision, write-back slot, dedup output and gathered byte.

Small workloads (every recipe, reduced) compare the full state after every
step; the full-size workloads run in the launch configuration the benchmark
times, with the oracle in id mode (exact: row contents are a function of the
address), full state compared every step and gathered bytes on sampled rows.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from synth.configs import WORKLOADS, small
from tests.harness import OracleRun, apply_events, check_invariants, check_step_outputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from tests.gpu_harness import (GpuReplay, check_gpu_internal, check_layer_signal, compare_states,
                                   expand_id_rows, gpu_state_in_oracle_terms)


def run_parity(w, steps, mode="bytes", state_every=1, out_every=1, sample_rows=2048, seed=0,
               group_streams=False):
    gpu = GpuReplay(w, group_streams=group_streams)
    orc = OracleRun(w, mode)
    rng = np.random.default_rng(seed)
    try:
        for g in range(w.n_groups):  # initial placement
            compare_states(gpu_state_in_oracle_terms(gpu.cache.export(g), w), orc.o.export(g),
                           f"initial g{g}", orc.o.stamps(g))
        for t in range(steps):
            sel, ev = gpu.trace.step()
            gpu.run_groups(sel)
            for g in range(w.n_groups):
                ro = orc.o.step_group(g, sel[g])
                full = (t % out_every == 0)
                rg = gpu.results(g, full_out=full and mode == "bytes")
                where = f"step {t} group {g}"
                assert np.array_equal(rg["req_off"], ro["req_off"]), where
                assert np.array_equal(rg["entry_row"], ro["entry_row"]), where
                U = int(ro["req_off"][-1])
                if full and mode == "bytes":
                    assert np.array_equal(rg["out"], ro["out"][:, :U]), f"{where}: gathered bytes"
                else:
                    rows = rng.choice(U, min(U, sample_rows), replace=False) if U else np.zeros(0, int)
                    rows_t = torch.from_numpy(rows).to(gpu.outs[g].device)
                    for j in range(w.layers_per_group):
                        got = gpu.outs[g][j].index_select(0, rows_t).cpu().numpy()
                        if mode == "bytes":
                            exp = ro["out"][j, rows]
                        else:
                            exp = expand_id_rows(ro["out"][j, rows], w.seed, g, j, w.row_bytes)
                        assert np.array_equal(got, exp), f"{where}: gathered bytes layer {j}"
                if w.layer_signal:
                    check_layer_signal(gpu.cache, g, w.layers_per_group, where)
                if t % state_every == 0 or t == steps - 1:
                    st = gpu.cache.export(g)
                    check_gpu_internal(st, w)
                    go = gpu_state_in_oracle_terms(st, w)
                    oo = orc.o.export(g)
                    compare_states(go, oo, where, orc.o.stamps(g))
                    v, vc, wb = orc.o.last_decisions(g)
                    assert st["M"] == len(v) and st["writebacks"] == len(wb), where
                    assert np.array_equal(st["victims"][:len(v)], v), f"{where}: victims"
                    assert np.array_equal(st["wb_host"][:len(wb)], wb), f"{where}: write-backs"
                    check_invariants(go, w.gpu_slots, w.host_slots, orc.live)
            from tests.harness import apply_events
            apply_events(gpu.alloc, gpu.free, ev)
            apply_events(orc.alloc, orc.free, ev)
        return gpu.cache.sync()
    finally:
        gpu.close()


def test_parity_tiny_1x4k_full():
    stats = run_parity(WORKLOADS["tiny_1x4k"], WORKLOADS["tiny_1x4k"].steps)
    assert stats["steps"] == 64 and stats["misses"] > 0 and stats["hits"] > 0


@pytest.mark.parametrize("name", ["batch8_32k", "longdoc", "low_evict", "low_overlap", "low_overlap_256"])
def test_parity_small(name):
    w = small(name)
    stats = run_parity(w, w.steps)
    assert stats["misses"] > 0
    if w.bypass:
        assert stats["bypassed"] > 0  # the literal recipe overflows the pool every step


def test_parity_batch8_32k_full():
    w = WORKLOADS["batch8_32k"]
    stats = run_parity(w, w.steps, mode="bytes", state_every=4, out_every=16)
    assert stats["steps"] == w.steps * w.n_groups and stats["writebacks"] > 0


@pytest.mark.parametrize("name,beside,exact", [("longdoc", False, False), ("low_overlap", False, False),
                                               ("low_overlap_256", True, False),
                                               ("low_evict", False, True), ("longdoc", True, True)])
def test_parity_small_group_streams(name, beside, exact):
    """Each group's call on its own caller stream: a group's metadata runs while earlier
    groups' copies (and, beside the move, gathers) are still running; same results."""
    w = small(name).replace(gather_beside=beside, exact_lru=exact)
    stats = run_parity(w, w.steps, group_streams=True)
    assert stats["misses"] > 0


@pytest.mark.parametrize("name,beside,exact", [("longdoc", False, False), ("low_overlap", False, False),
                                               ("longdoc", True, False), ("low_evict", False, True)])
def test_pipelined_steps_match_oracle(name, beside, exact):
    """Steps issued ahead with no synchronisation between them, as the benchmark issues
    them: each group's calls on its own caller stream, each step's alloc/free on the main
    stream (rows in buffers of their own), per-step outputs.  After one final sync, every
    step's outputs and the final state equal the oracle's."""
    from oracle.replay import alloc_rows
    w = small(name).replace(gather_beside=beside, exact_lru=exact)
    n = 12
    gpu = GpuReplay(w, group_streams=True)
    orc = OracleRun(w, "bytes")
    G, E, R = w.n_groups, w.entries_per_step, w.n_live
    dev = gpu.cache.device
    try:
        sels, evs = [], []
        for _ in range(n):
            sel, ev = gpu.trace.step()
            sels.append(sel)
            evs.append(ev)
        sel_d = torch.from_numpy(np.stack(sels).view(np.int32)).to(dev)
        torch.cuda.synchronize()
        outs = [[gpu.cache.out_buffer(g, E) for g in range(G)] for _ in range(n)]
        ers = [[torch.empty(E, dtype=torch.int32, device=dev) for _ in range(G)] for _ in range(n)]
        ros = [[torch.empty(R + 1, dtype=torch.int32, device=dev) for _ in range(G)] for _ in range(n)]
        keep = []

        def dev_alloc(base, m):
            rows = torch.from_numpy(alloc_rows(w, base, m, "bytes")).pin_memory()
            keep.append(rows)
            return gpu.cache.alloc(m, rows)

        for t in range(n):
            for g in range(G):
                gpu.cache.step_group(g, sel_d[t, g], outs[t][g], ers[t][g], ros[t][g],
                                     stream=gpu.gstreams[g])
            apply_events(dev_alloc, gpu.cache.free, evs[t])
        gpu.cache.sync()
        torch.cuda.synchronize()
        for t in range(n):
            for g in range(G):
                ro = orc.o.step_group(g, sels[t][g])
                where = f"step {t} group {g}"
                assert np.array_equal(ros[t][g].cpu().numpy(), ro["req_off"]), where
                assert np.array_equal(ers[t][g].cpu().numpy(), ro["entry_row"]), where
                U = int(ro["req_off"][-1])
                assert np.array_equal(outs[t][g][:, :U].cpu().numpy(), ro["out"][:, :U]), where
            apply_events(orc.alloc, orc.free, evs[t])
        for g in range(G):
            st = gpu.cache.export(g)
            check_gpu_internal(st, w)
            compare_states(gpu_state_in_oracle_terms(st, w), orc.o.export(g), f"final g{g}",
                           orc.o.stamps(g))
    finally:
        gpu.close()


@pytest.mark.parametrize("name", ["longdoc", "low_overlap_256"])
def test_parity_small_gather_beside_move(name):
    """The hit gather beside the move (ULA_FLAG_GATHER_BESIDE_MOVE): same results."""
    w = small(name).replace(gather_beside=True)
    stats = run_parity(w, w.steps)
    assert stats["misses"] > 0


def test_parity_full_size_sampled_gather_beside_move():
    w = WORKLOADS["longdoc"].replace(gather_beside=True)
    stats = run_parity(w, 6, mode="id", state_every=1, out_every=10**9, sample_rows=4096,
                       group_streams=True)
    assert stats["steps"] == 6 * w.n_groups


@pytest.mark.parametrize("beside", [False, True])
def test_copy_kernel_spans(beside):
    """Every step records one span per copy kernel (gather, staging, move) and one for its
    metadata (dedup through victim emission), each with a start no later than its end,
    in launch order; by default the move starts after the gather ended."""
    from serving_step_sparse_gb300 import ula
    w = small("longdoc").replace(steps=6, gather_beside=beside)
    gpu = GpuReplay(w)
    try:
        gpu.step()
        ula.ula_profile_spans(gpu.cache.ctx, True)
        n = 3
        for _ in range(n):
            gpu.step()
        spans = ula.ula_profile_spans_read(gpu.cache.ctx)
        ula.ula_profile_spans(gpu.cache.ctx, False)
        assert ula.ula_profile_spans_read(gpu.cache.ctx) == []  # read clears
        kinds = [(ph, g) for ph, g, _, _ in spans]
        for g in range(w.n_groups):
            for ph in ("select", "gather", "stage", "move"):  # select: dedup .. victim emission
                assert kinds.count((ph, g)) == n, (ph, g)
        for ph, g, t0, t1 in spans:
            assert 0 < t0 <= t1, (ph, g, t0, t1)
        per = {}
        for ph, g, t0, t1 in spans:
            per.setdefault(g, []).append((ph, t0, t1))
        for g, lst in per.items():  # per group step: its four records, the move's last
            for i in range(0, len(lst), 4):
                rec = {ph: (t0, t1) for ph, t0, t1 in lst[i:i + 4]}
                assert sorted(rec) == ["gather", "move", "select", "stage"], lst[i:i + 4]
                assert lst[i][0] == "select" and lst[i + 3][0] == "move"
                (q0, q1), (g0, g1), (s0, s1), (m0, m1) = (rec[k] for k in ("select", "gather",
                                                                          "stage", "move"))
                assert g0 >= q0 and s0 >= q1 and m0 >= q1 and m0 >= s1
                if not beside:
                    assert m0 >= g1, "the move starts after the hit gather"
    finally:
        gpu.close()


# ----------------------------------------------------------------- edge cases

def test_pads_and_ragged_sizes():
    # ragged: S, H not multiples of 32 or 1,024; E not a multiple of the block size
    w = WORKLOADS["tiny_1x4k"].replace(pad_prob=0.1, gpu_slots_explicit=1000 + 7,
                                  host_slots_explicit=3400 + 13, k=250, window=50, steps=32)
    assert w.gpu_slots + w.host_slots >= w.max_live_history + w.entries_per_step
    run_parity(w, w.steps)


@pytest.mark.parametrize("B", [1, 2, 3])
def test_small_rings(B):
    w = small("batch8_32k").replace(ring_buckets=B, steps=24)
    run_parity(w, w.steps)


def test_everything_fits_on_gpu_no_host_pool():
    w = WORKLOADS["tiny_1x4k"].replace(gpu_slots_explicit=4096, host_slots_explicit=0, steps=16)
    stats = run_parity(w, w.steps)
    assert stats["misses"] == 0 and stats["writebacks"] == 0


def _direct(S=64, H=256, B=3, layers=(1, 3), W=16, max_logical=512, max_entries=64,
            exact=False):
    from serving_step_sparse_gb300.cache import UlaCache
    from oracle import Oracle
    c = UlaCache(row_bytes=W, layers_per_group=list(layers), gpu_slots=S, host_slots=H,
                 ring_buckets=B, max_logical=max_logical, max_entries=max_entries,
                 exact_lru=exact)
    o = Oracle(W, list(layers), S, H, B, max_logical, exact_lru=exact)
    return c, o


def _rows(layers, base, n, W, seed=9):
    parts = [synth.content_range(seed, g, L, base, n, W).reshape(-1) for g, L in enumerate(layers)]
    return np.concatenate(parts)


def _step_both(c, o, g, sel, cap=None):
    from tests.gpu_harness import gpu_state_in_oracle_terms
    sel = np.ascontiguousarray(sel, dtype=np.uint32)
    R, Q, K = sel.shape
    cap = cap if cap is not None else max(1, sel.size)
    out = c.out_buffer(g, cap)
    er = torch.empty(max(1, sel.size), dtype=torch.int32, device="cuda")
    ro = torch.empty(R + 1, dtype=torch.int32, device="cuda")
    sd = torch.from_numpy(sel.view(np.int32).copy()).cuda()
    c.step_group(g, sd, out, er, ro)
    c.sync()
    res = o.step_group(g, sel, out_cap=cap)
    U = int(res["req_off"][-1])
    assert np.array_equal(ro.cpu().numpy(), res["req_off"])
    assert np.array_equal(er.cpu().numpy()[:sel.size], res["entry_row"])
    assert np.array_equal(out[:, :U].cpu().numpy(), res["out"][:, :U])
    return res


class _W:  # geometry shim for the state converters
    def __init__(self, S, H, B):
        self.gpu_slots, self.host_slots, self.ring_buckets = S, H, B


def test_mixed_layers_duplicates_across_requests_and_empty_steps():
    from tests.gpu_harness import gpu_state_in_oracle_terms
    layers, W, S, H, B = (1, 3), 16, 64, 256, 3
    c, o = _direct(S=S, H=H, B=B, layers=layers, W=W)
    try:
        n = 200
        rows = _rows(layers, 0, n, W)
        t = torch.from_numpy(rows).pin_memory()
        assert c.alloc(n, t) == 0 and o.alloc(n, rows) == 0
        c.sync()
        rng = np.random.default_rng(3)
        for step in range(40):
            g = step % 2
            if step % 7 == 3:  # empty selections: no requests, or k = 0
                _step_both(c, o, g, np.zeros((0, 1, 4), np.uint32))
                _step_both(c, o, g, np.zeros((2, 1, 0), np.uint32))
                continue
            R, Q, K = 3, 2, 8
            sel = rng.choice(n, (R, Q, K)).astype(np.uint32)
            sel[1, 0, :4] = sel[0, 1, :4]  # the same addresses in two requests
            sel[2, 1, 3] = 0xFFFFFFFF
            _step_both(c, o, g, sel)
            for gg in range(2):
                go = gpu_state_in_oracle_terms(c.export(gg), _W(S, H, B))
                compare_states(go, o.export(gg), f"step {step} g{gg}")
    finally:
        c.close()


def test_bulk_and_register_gathers_by_row_length():
    """Group 0's rows (2 layers x 656 B) fit the bulk gather's per-thread buffers; group 1's
    (10 layers x 656 B = 6,560 B) do not and take the register gather.  Both, and the moves
    beside them, bit-exact with the oracle over steps with evictions in both groups."""
    from tests.gpu_harness import gpu_state_in_oracle_terms
    layers, W, S, H, B = (2, 10), 656, 48, 512, 3
    c, o = _direct(S=S, H=H, B=B, layers=layers, W=W, max_logical=512, max_entries=256)
    try:
        n = 400
        rows = _rows(layers, 0, n, W)
        t = torch.from_numpy(rows).pin_memory()
        assert c.alloc(n, t) == 0 and o.alloc(n, rows) == 0
        c.sync()
        rng = np.random.default_rng(11)
        misses = writebacks = 0
        for step in range(24):
            g = step % 2
            sel = rng.choice(n, (2, 2, 8)).astype(np.uint32)  # at most 32 unique rows (S = 48)
            sel[1, 1, 5] = 0xFFFFFFFF
            res = _step_both(c, o, g, sel)
            misses += res["counters"]["misses"]
            writebacks += res["counters"]["writebacks"]
            for gg in range(2):
                go = gpu_state_in_oracle_terms(c.export(gg), _W(S, H, B))
                compare_states(go, o.export(gg), f"step {step} g{gg}")
        assert misses > 0 and writebacks > 0
    finally:
        c.close()


# --------------------------------------------------------- per-layer signal

@pytest.mark.parametrize("name", ["tiny_1x4k", "batch8_32k", "longdoc", "low_overlap",
                                  "low_overlap_256"])
def test_layer_signal_parity_small(name):
    """Layer-major fill with per-layer flags: outputs and state bit-exact with the
    oracle, every flag at the step's round after the step."""
    w = (WORKLOADS[name] if name == "tiny_1x4k" else small(name)).replace(layer_signal=True)
    stats = run_parity(w, min(w.steps, 24))
    assert stats["misses"] > 0


@pytest.mark.parametrize("name,steps", [("longdoc", 6), ("low_overlap_256", 4)])
def test_layer_signal_full_size_sampled(name, steps):
    w = WORKLOADS[name].replace(layer_signal=True)
    run_parity(w, steps, mode="id", state_every=1, out_every=10**9, sample_rows=4096)


def test_layer_signal_consumers_on_another_stream():
    """Model consumers of every layer, launched on another stream right after each
    group call and before any synchronisation, each wait for their layer's flag and
    read exactly the oracle's rows for that layer."""
    from serving_step_sparse_gb300 import ula
    from tests.harness import apply_events
    w = WORKLOADS["batch8_32k"].replace(layer_signal=True, steps=10)
    gpu = GpuReplay(w)
    orc = OracleRun(w, "bytes")
    L = w.layers_per_group
    side = torch.cuda.Stream()
    res = torch.zeros((w.n_groups, L, 3), dtype=torch.int64, device="cuda")
    early = total = 0
    try:
        for t in range(w.steps):
            sel, ev = gpu.trace.step()
            gpu.sel_d.copy_(torch.from_numpy(np.ascontiguousarray(sel).view(np.int32)))
            for g in range(w.n_groups):
                gpu.cache.step_group(g, gpu.sel_d[g], gpu.outs[g], gpu.entry_row[g], gpu.req_off[g])
                _, rnd = gpu.cache.layer_signal(g)
                ro = orc.o.step_group(g, sel[g])
                U = int(ro["req_off"][-1])
                for j in range(L):
                    ula.ula_debug_consume(gpu.cache.ctx, g, j, rnd, gpu.outs[g].data_ptr(),
                                          gpu.cap, U, res[g, j].data_ptr(), side.cuda_stream)
                exp = [int(ro["out"][j, :U].view(np.uint32).sum(dtype=np.uint64) & 0xFFFFFFFF)
                       for j in range(L)]
                torch.cuda.synchronize()
                gpu.cache.sync()
                r = res[g].cpu().numpy().astype(np.uint64)
                ns = ula.ula_debug_layer_times(gpu.cache.ctx, g, L)
                for j in range(L):
                    assert r[j, 2] == 0, f"step {t} group {g} layer {j}: consumer timed out"
                    assert int(r[j, 1]) == exp[j], f"step {t} group {g} layer {j}: checksum"
                    assert r[j, 0] >= ns[j]  # it saw the flag after the flag was set
                total += 1
                early += int(r[0, 0] < ns[L - 1])  # layer 0 read before the last layer landed
            apply_events(gpu.alloc, gpu.free, ev)
            apply_events(orc.alloc, orc.free, ev)
        print(f"layer-0 consumer started before the last layer was signalled in {early}/{total}")
    finally:
        gpu.close()


def test_layer_signal_with_exact_lru():
    w = small("low_evict").replace(layer_signal=True, exact_lru=True, steps=24)
    run_parity(w, w.steps)


# ----------------------------------------------------------------- exact LRU

@pytest.mark.parametrize("name", ["batch8_32k", "longdoc", "low_evict", "low_overlap", "low_overlap_256"])
def test_exact_lru_parity_small(name):
    w = small(name).replace(exact_lru=True)
    stats = run_parity(w, w.steps)
    assert stats["misses"] > 0 and stats["victims_cold"] > 0 and stats["victims_ring"] == 0


@pytest.mark.parametrize("name,steps", [("longdoc", 8), ("low_evict", 8), ("low_overlap_256", 4)])
def test_exact_lru_full_size_sampled(name, steps):
    w = WORKLOADS[name].replace(exact_lru=True)
    stats = run_parity(w, steps, mode="id", state_every=1, out_every=10**9, sample_rows=4096)
    assert stats["steps"] == steps * w.n_groups


def test_exact_lru_wide_timestamp_spread():
    """Timestamps thousands of rounds apart: a two-digit radix select and a two-pass
    sort of the chosen slots (their keys span more than 256 rounds)."""
    from tests.gpu_harness import gpu_state_in_oracle_terms
    layers, W, S, H, B = (1,), 16, 64, 512, 8
    c, o = _direct(S=S, H=H, B=B, layers=layers, W=W, max_logical=1024, max_entries=64,
                   exact=True)
    try:
        n = 400
        rows = _rows(layers, 0, n, W)
        assert c.alloc(n, torch.from_numpy(rows).pin_memory()) == 0 and o.alloc(n, rows) == 0
        c.sync()
        hot = np.arange(0, 16, dtype=np.uint32)           # touched every round
        warm = np.arange(16, 40, dtype=np.uint32)         # one touched every 120 rounds
        cold = np.arange(64, n, dtype=np.uint32)          # on the host, pulled in bursts
        rng = np.random.default_rng(5)
        rounds = 3200
        bursts = 0
        wide = []  # (candidate timestamp span, chosen victims' timestamp span) per burst
        for step in range(rounds):
            sel = [hot]
            if step % 120 == 0:
                sel.append(warm[(step // 120) % len(warm):][:1])
            if step in (1500, 2600, 3100, 3199):
                sel.append(rng.choice(cold, 20, replace=False).astype(np.uint32))
                bursts += 1
            flat = np.concatenate(sel)
            if step in (1500, 2600, 3100, 3199) or step % 400 == 0:
                before, _ = o.stamps(0)
                _step_both(c, o, 0, flat.reshape(1, 1, -1))
                go = gpu_state_in_oracle_terms(c.export(0), _W(S, H, B))
                compare_states(go, o.export(0), f"round {step}", o.stamps(0))
                v, vc, wb = o.last_decisions(0)
                st = c.export(0)
                assert np.array_equal(st["victims"][:len(v)], v), f"round {step}: victims"
                if len(v):
                    occ = before[before != 0xFFFFFFFF]
                    wide.append((int(occ.max() - occ.min()),
                                 int(before[v].max()) - int(before[v].min())))
            else:  # quick rounds: GPU and oracle step, outputs not compared
                sd = torch.from_numpy(flat.view(np.int32).copy()).cuda()
                out = c.out_buffer(0, flat.size)
                er = torch.empty(flat.size, dtype=torch.int32, device="cuda")
                ro = torch.empty(2, dtype=torch.int32, device="cuda")
                c.step_group(0, sd.view(1, 1, -1), out, er, ro)
                o.step_group(0, flat.reshape(1, 1, -1))
        assert bursts == 4 and o.stamps(0)[1] == rounds
        assert any(a >= 2048 and b >= 256 for a, b in wide), wide
        c.sync()
    finally:
        c.close()


def test_exact_lru_general_path_when_the_window_runs_short():
    """The fast scan bins timestamps within 2,047 rounds of a lower bound kept from the
    previous scan; when fewer than Q candidates lie in that window (a few slots left
    untouched for thousands of rounds, the rest recent) the general path runs: an exact
    oldest-stamp scan, a 32-bit radix select and a stable sort."""
    from tests.gpu_harness import gpu_state_in_oracle_terms
    layers, W, S, H, B = (1,), 16, 64, 512, 8
    c, o = _direct(S=S, H=H, B=B, layers=layers, W=W, max_logical=1024, max_entries=64,
                   exact=True)
    try:
        n = 300
        rows = _rows(layers, 0, n, W)
        assert c.alloc(n, torch.from_numpy(rows).pin_memory()) == 0 and o.alloc(n, rows) == 0
        c.sync()
        rng = np.random.default_rng(8)
        bursts = [(2600, 20), (2601, 3), (5000, 40)]
        for step in range(5001):
            if step < 2100:
                flat = np.array([60, 61, 62, 63], dtype=np.uint32)  # resident, always hits
            else:  # touch 5..63 a few at a time; 0..4 stay at their first stamp
                flat = np.unique(np.concatenate([[60, 61, 62, 63],
                                                 rng.choice(np.arange(5, 64), 3, replace=False)]))
                flat = flat.astype(np.uint32)
            burst = dict(bursts).get(step)
            if burst:
                flat = np.concatenate([flat, rng.choice(np.arange(64, n), burst, replace=False)
                                       .astype(np.uint32)])
                flat = np.unique(flat).astype(np.uint32)
                _step_both(c, o, 0, flat.reshape(1, 1, -1))
                go = gpu_state_in_oracle_terms(c.export(0), _W(S, H, B))
                compare_states(go, o.export(0), f"round {step}", o.stamps(0))
                v, vc, wb = o.last_decisions(0)
                assert np.array_equal(c.export(0)["victims"][:len(v)], v), f"round {step}"
            else:
                sd = torch.from_numpy(flat.view(np.int32).copy()).cuda()
                out = c.out_buffer(0, flat.size)
                er = torch.empty(flat.size, dtype=torch.int32, device="cuda")
                ro = torch.empty(2, dtype=torch.int32, device="cuda")
                c.step_group(0, sd.view(1, 1, -1), out, er, ro)
                o.step_group(0, flat.reshape(1, 1, -1))
        st = c.sync()
        assert st["victims_cold"] > 0
    finally:
        c.close()


def test_exact_lru_barrier_wait_is_bounded():
    """A block that never arrives at the scan's grid-wide barrier (test hook): the
    others give up after their bound, the step reports ULA_ERR_TIMEOUT and the
    context refuses further work; the GPU stays usable."""
    import time
    from serving_step_sparse_gb300 import ula
    layers, W, S, H, B = (1,), 16, 64, 512, 4
    c, o = _direct(S=S, H=H, B=B, layers=layers, W=W, max_logical=1024, max_entries=64,
                   exact=True)
    try:
        n = 200
        rows = _rows(layers, 0, n, W)
        assert c.alloc(n, torch.from_numpy(rows).pin_memory()) == 0
        c.sync()
        sel = np.arange(100, 120, dtype=np.uint32).reshape(1, 1, -1)  # 20 misses, no free slot
        out = c.out_buffer(0, 20)
        er = torch.empty(20, dtype=torch.int32, device="cuda")
        ro = torch.empty(2, dtype=torch.int32, device="cuda")
        sd = torch.from_numpy(sel.view(np.int32).copy()).cuda()
        ula.ula_debug_inject(c.ctx, ula.DEBUG_STALL_SCAN_BARRIER)
        t0 = time.monotonic()
        c.step_group(0, sd, out, er, ro)
        with pytest.raises(ula.UlaError) as ei:
            c.sync()
        assert ei.value.code == ula.ERR_TIMEOUT
        assert time.monotonic() - t0 < 20.0
        with pytest.raises(ula.UlaError) as ei:
            c.step_group(0, sd, out, er, ro)
        assert ei.value.code == ula.ERR_POISONED
    finally:
        c.close()
    x = torch.ones(1 << 20, device="cuda")  # the device still runs work
    assert float(x.sum()) == float(1 << 20)


def _export_all(c, G, S, H, B):
    from tests.gpu_harness import gpu_state_in_oracle_terms
    return [gpu_state_in_oracle_terms(c.export(g), _W(S, H, B)) for g in range(G)]


def _same(a, b):
    return all(all(np.array_equal(x[k], y[k]) for k in x if k in y) for x, y in zip(a, b))


@pytest.mark.parametrize("case", ["capacity", "unmapped", "out_cap", "inject"])
def test_device_errors_latch_poison_and_change_nothing(case):
    from serving_step_sparse_gb300 import ula
    S, H, B, layers, W = 32, 128, 4, (2,), 32
    c, o = _direct(S=S, H=H, B=B, layers=layers, W=W, max_logical=256, max_entries=64)
    try:
        n = 100
        t = torch.from_numpy(_rows(layers, 0, n, W)).pin_memory()
        c.alloc(n, t)
        c.sync()
        before = _export_all(c, 1, S, H, B)
        if case == "capacity":   # 33 distinct addresses > 32 GPU slots
            sel = np.arange(33, dtype=np.uint32).reshape(1, 1, 33)
            cap, want = 64, ula.ERR_CAPACITY
        elif case == "unmapped":  # address 150 was never allocated
            sel = np.array([[[1, 2, 150]]], dtype=np.uint32)
            cap, want = 64, ula.ERR_UNMAPPED
        elif case == "out_cap":
            sel = np.arange(10, dtype=np.uint32).reshape(1, 1, 10)
            cap, want = 9, ula.ERR_CAPACITY
        else:
            c.inject(ula.ERR_TIMEOUT)
            sel = np.arange(4, dtype=np.uint32).reshape(1, 1, 4)
            cap, want = 64, ula.ERR_TIMEOUT
        sd = torch.from_numpy(sel.view(np.int32).copy()).cuda()
        out = c.out_buffer(0, cap)
        er = torch.empty(sel.size, dtype=torch.int32, device="cuda")
        ro = torch.empty(2, dtype=torch.int32, device="cuda")
        c.step_group(0, sd, out, er, ro)
        assert ula.ula_sync_rc(c.ctx) == want
        after = _export_all(c, 1, S, H, B)
        # the round counter advanced on the host, but no label, map entry or slot changed
        for x, y in zip(before, after):
            for k in ("tier", "slot", "cls", "owner", "host_free", "host_owner"):
                assert np.array_equal(x[k], y[k]), k
        with pytest.raises(ula.UlaError) as ei:
            c.step_group(0, sd, out, er, ro)
        assert ei.value.code == ula.ERR_POISONED
        with pytest.raises(ula.UlaError) as ei:
            c.sync()
        assert ei.value.code == ula.ERR_POISONED
    finally:
        c.close()


def test_host_detected_errors_change_nothing():
    from serving_step_sparse_gb300 import ula
    S, H, B, layers, W = 16, 16, 2, (1,), 16
    c, o = _direct(S=S, H=H, B=B, layers=layers, W=W, max_logical=64, max_entries=8)
    try:
        t = torch.from_numpy(_rows(layers, 0, 20, W)).pin_memory()
        assert c.alloc(20, t) == 0
        c.sync()
        before = _export_all(c, 1, S, H, B)
        big = torch.from_numpy(_rows(layers, 20, 13, W)).pin_memory()
        with pytest.raises(ula.UlaError) as ei:  # 20 + 13 > S + H
            c.alloc(13, big)
        assert ei.value.code == ula.ERR_CAPACITY
        pageable = torch.zeros(16, dtype=torch.uint8)
        with pytest.raises(ula.UlaError) as ei:
            ula.ula_alloc(c.ctx, 1, pageable.data_ptr())
        assert ei.value.code == ula.ERR_INVALID_ARG
        c.free(3, 2)
        with pytest.raises(ula.UlaError) as ei:  # double free
            c.free(4, 1)
        assert ei.value.code == ula.ERR_INVALID_ARG
        with pytest.raises(ula.UlaError) as ei:  # beyond what was allocated
            c.free(19, 2)
        assert ei.value.code == ula.ERR_INVALID_ARG
        sd = torch.zeros((1, 1, 9), dtype=torch.int32, device="cuda")
        out = c.out_buffer(0, 9)
        er = torch.empty(9, dtype=torch.int32, device="cuda")
        ro = torch.empty(2, dtype=torch.int32, device="cuda")
        with pytest.raises(ula.UlaError) as ei:  # 9 entries > max_entries
            c.step_group(0, sd, out, er, ro)
        assert ei.value.code == ula.ERR_INVALID_ARG
        with pytest.raises(ula.UlaError) as ei:
            ula.ula_step_group(c.ctx, 1, sd.data_ptr(), 1, 1, 1, out.data_ptr(), 9,
                               er.data_ptr(), ro.data_ptr(), None, c.stream.cuda_stream)
        assert ei.value.code == ula.ERR_INVALID_ARG
        c.sync()  # still healthy
        after = _export_all(c, 1, S, H, B)
        o.alloc(20, _rows(layers, 0, 20, W))
        o.free(3, 2)
        assert _same(after, [o.export(0)])
        assert before[0]["tier"][3] != 0 and after[0]["tier"][3] == 0
    finally:
        c.close()


def test_config_and_pool_validation():
    from serving_step_sparse_gb300 import ula
    gp = torch.empty(4 * 16, dtype=torch.uint8, device="cuda")
    hp = torch.empty(4 * 16, dtype=torch.uint8, pin_memory=True)
    good = dict(row_bytes=16, layers_per_group=[1], gpu_slots=4, host_slots=4, ring_buckets=2,
                max_logical=8, max_entries=4)
    for bad in (dict(row_bytes=20), dict(ring_buckets=0), dict(ring_buckets=65), dict(gpu_slots=0),
                dict(max_entries=0), dict(layers_per_group=[0])):
        cfg = ula.make_config(**{**good, **bad})
        with pytest.raises(ula.UlaError) as ei:
            ula.ula_create(cfg, [gp.data_ptr()], [hp.data_ptr()], None)
        assert ei.value.code == ula.ERR_INVALID_ARG
    cfg = ula.make_config(**good)
    pageable = torch.empty(64, dtype=torch.uint8)
    with pytest.raises(ula.UlaError):  # host pool must be pinned
        ula.ula_create(cfg, [gp.data_ptr()], [pageable.data_ptr()], None)
    with pytest.raises(ula.UlaError):  # GPU pool must be device memory
        ula.ula_create(cfg, [hp.data_ptr()], [hp.data_ptr()], None)
    with pytest.raises(ula.UlaError):  # 16-byte alignment
        ula.ula_create(cfg, [gp.data_ptr() + 8], [hp.data_ptr()], None)
    ctx = ula.ula_create(cfg, [gp.data_ptr()], [hp.data_ptr()], None)
    ula.ula_destroy(ctx)


def test_layer_ready_events_and_side_stream_order():
    """Layer j's event completes after its rows are written; a consumer waiting on
    each event (on another stream) reads the right bytes."""
    w = small("batch8_32k").replace(steps=6)
    gpu = GpuReplay(w)
    orc = OracleRun(w, "bytes")
    consumer = torch.cuda.Stream()
    try:
        for t in range(w.steps):
            sel, ev = gpu.trace.step()
            gpu.sel_d.copy_(torch.from_numpy(sel.view(np.int32)))
            copies = []
            for g in range(w.n_groups):
                events = [torch.cuda.Event() for _ in range(w.layers_per_group)]
                gpu.cache.step_group(g, gpu.sel_d[g], gpu.outs[g], gpu.entry_row[g],
                                     gpu.req_off[g], layer_ready=events)
                with torch.cuda.stream(consumer):
                    for j, e in enumerate(events):
                        consumer.wait_event(e)
                        copies.append((g, j, gpu.outs[g][j].clone()))
            consumer.synchronize()
            gpu.cache.sync()
            for g in range(w.n_groups):
                ro = orc.o.step_group(g, sel[g])
                U = int(ro["req_off"][-1])
                for gg, j, buf in copies:
                    if gg == g:
                        assert np.array_equal(buf[:U].cpu().numpy(), ro["out"][j, :U])
            from tests.harness import apply_events
            apply_events(gpu.alloc, gpu.free, ev)
            apply_events(orc.alloc, orc.free, ev)
    finally:
        gpu.close()


def test_regather_reproduces_hit_rows():
    """ula_debug_regather (used to time the gather alone) writes the same hit rows."""
    from serving_step_sparse_gb300 import ula
    w = small("batch8_32k").replace(steps=5)
    gpu = GpuReplay(w)
    try:
        for _ in range(w.steps):
            gpu.step()
        for g in range(w.n_groups):
            st = gpu.cache.export(g)
            U = st["U"]
            hit = st["row_slot"][:U] != 0xFFFFFFFF
            assert hit.sum() == st["hits"]
            for j in range(w.layers_per_group):
                buf = torch.zeros_like(gpu.outs[g])
                ula.ula_debug_regather(gpu.cache.ctx, g, j, buf.data_ptr(), buf.shape[1],
                                       torch.cuda.current_stream().cuda_stream,
                                       blocks_per_sm=2 if j % 2 else 0)
                torch.cuda.synchronize()
                got = buf[j, :U].cpu().numpy()[hit]
                exp = gpu.outs[g][j, :U].cpu().numpy()[hit]
                assert np.array_equal(got, exp)
            # layer ranges in one launch (the step gathers every layer in one)
            L = w.layers_per_group
            for j0, n in ((1, L - 1), (0, L), (0, L - 1)):
                buf = torch.zeros_like(gpu.outs[g])
                ula.ula_debug_regather(gpu.cache.ctx, g, j0, buf.data_ptr(), buf.shape[1],
                                       torch.cuda.current_stream().cuda_stream,
                                       blocks_per_sm=2 if j0 else 0, n_layers=n)
                torch.cuda.synchronize()
                got = buf[:, :U].cpu().numpy()
                exp = gpu.outs[g][:, :U].cpu().numpy()
                for j in range(L):
                    if j0 <= j < j0 + n:
                        assert np.array_equal(got[j][hit], exp[j][hit]), (j0, n, j)
                    else:
                        assert not got[j].any(), (j0, n, j)  # other layers untouched
            with pytest.raises(ula.UlaError):
                ula.ula_debug_regather(gpu.cache.ctx, g, 1, buf.data_ptr(), buf.shape[1],
                                       torch.cuda.current_stream().cuda_stream, n_layers=L)
        # into a buffer shorter than the step's unique rows: the gather latches the capacity
        # error on the device (and writes nothing), the next sync reports it
        U = gpu.cache.export(0)["U"]
        short = gpu.cache.out_buffer(0, max(1, U - 1))
        ula.ula_debug_regather(gpu.cache.ctx, 0, 0, short.data_ptr(), short.shape[1],
                               torch.cuda.current_stream().cuda_stream, n_layers=w.layers_per_group)
        assert ula.ula_sync_rc(gpu.cache.ctx) == ula.ERR_CAPACITY
    finally:
        gpu.close()
