"""Pins of the CPU oracle against what the UlaCache summary page and plain
reasoning fix -- independent of the oracle's own code:

* a hand-worked PB-LRU example (tests/golden/pblru_worked_example.txt, §3 "PB-LRU");
* a special case that reduces to a textbook routine: with more ring buckets than
  rounds no fold can happen, and PB-LRU must evict exactly like round-granular
  LRU with the lowest slot first inside a round;
* with folds, a brute-force model written from per-slot timestamps (a slot is cold
  iff its last access is at least B rounds old) instead of bucket sets;
* the exact-LRU mode (§3's baseline policy: a timestamp per slot, the oldest
  evicted first) against the same brute force's round-granular LRU order, for any
  number of ring buckets, and the per-slot timestamps against the brute force's;
* the gathered rows against the generator's closed form (byte for byte);
* invariants: one tier per entry (§2), slot ownership, class partition, the
  current round's slots never evicted (§3), rotation changes labels only (§3),
  errors leave the state untouched.
"""
from __future__ import annotations

import os
import random

import numpy as np
import pytest

import synth
from oracle import (CAPACITY, COLD, FREE, INVALID_ARG, TIER_GPU, TIER_HOST, TIER_UNALLOCATED,
                    UNMAPPED, ExactLru, Oracle, OracleError)
from synth.configs import WORKLOADS, small
from tests.harness import (ID_ROW_BYTES, OracleRun, alloc_rows, check_invariants,
                           check_step_outputs, id_rows)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- golden example

def _parse_golden(path):
    cmds = []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                cmds.append(line.split())
    return cmds


def _id_row_buf(addr0, n):
    return id_rows(0, 1, addr0, n).reshape(-1)


def test_worked_example_golden():
    cmds = _parse_golden(os.path.join(GOLDEN, "pblru_worked_example.txt"))
    assert cmds[0][0] == "config"
    kv = dict(x.split("=") for x in cmds[0][1:])
    S, H, B, L = (int(kv[x]) for x in ("S", "H", "B", "L"))
    o = Oracle(ID_ROW_BYTES, [L], S, H, B, 64)
    last = None
    n_checks = 0
    for c in cmds[1:]:
        op = c[0]
        if op == "alloc":
            n, base = int(c[1]), int(c[3])
            assert o.alloc(n, _id_row_buf(base, n)) == base
        elif op == "free":
            o.free(int(c[1]), int(c[2]))
        elif op == "step":
            sel = np.array([int(x) for x in c[1:]], dtype=np.uint32).reshape(1, 1, -1)
            last = o.step_group(0, sel)
            # the gathered ids are the selected addresses (closed form)
            got = last["out"][0, :len(c) - 1].view(np.uint32)[:, 0]
            assert list(got) == [int(x) for x in c[1:]]
        elif op == "expect":
            what, vals = c[1], c[2:]
            st = o.export(0)
            n_checks += 1
            if what == "map":
                for v in vals:
                    a, loc = v.split(":")
                    a = int(a)
                    tier = TIER_GPU if loc[0] == "G" else TIER_HOST
                    assert st["tier"][a] == tier and st["slot"][a] == int(loc[1:]), v
            elif what == "unallocated":
                for v in vals:
                    assert st["tier"][int(v)] == TIER_UNALLOCATED
            elif what == "classes":
                for v in vals:
                    s, lab = v.split(":")
                    want = FREE if lab == "free" else COLD if lab == "cold" else int(lab[1:])
                    assert st["cls"][int(s)] == want, (v, st["cls"])
            elif what == "host_free":
                assert sorted(np.nonzero(st["host_free"])[0].tolist()) == [int(x) for x in vals]
            elif what == "victims":
                v, _, _ = o.last_decisions(0)
                assert v.tolist() == [int(x) for x in vals]
            elif what == "writeback":
                _, _, wb = o.last_decisions(0)
                assert wb.tolist() == [int(x) for x in vals]
            else:
                raise AssertionError(f"unknown expectation {what}")
    assert n_checks >= 25


# ------------------------------------------------------- brute-force reference

class BruteForce:
    """Residency by per-slot timestamps (not bucket sets).

    PB-LRU's eviction order, stated with timestamps: free slots ascending; then
    slots whose last access is at least B rounds old (the cold bucket), ascending;
    then, round by round from the oldest ring round to the previous one, the slots
    last accessed in that round, ascending.  With lru=True the order is plain
    round-granular LRU: free ascending, then occupied slots by (last round, slot).
    """

    def __init__(self, S, H, B, lru=False, bypass=False):
        self.S, self.H, self.B, self.lru, self.bypass = S, H, B, lru, bypass
        self.loc = {}          # addr -> ("G"|"H", slot)
        self.owner = {}        # GPU slot -> addr
        self.host_owner = {}   # host slot -> addr
        self.last = {}         # GPU slot -> last round accessed
        self.round = 0
        self.next = 0

    def alloc(self, n):
        base = self.next
        for a in range(base, base + n):
            free = [s for s in range(self.S) if s not in self.owner]
            if free:
                s = free[0]
                self.owner[s], self.last[s], self.loc[a] = a, self.round, ("G", s)
            else:
                h = min(x for x in range(self.H) if x not in self.host_owner)
                self.host_owner[h], self.loc[a] = a, ("H", h)
        self.next += n
        return base

    def free(self, base, n):
        for a in range(base, base + n):
            t, s = self.loc.pop(a)
            if t == "G":
                del self.owner[s], self.last[s]
            else:
                del self.host_owner[s]

    def order(self):
        free = [s for s in range(self.S) if s not in self.owner]
        occ = [s for s in self.owner if self.last[s] != self.round]
        if self.lru:
            return free + sorted(occ, key=lambda s: (self.last[s], s))
        r, B = self.round, self.B
        cold = sorted(s for s in occ if self.last[s] <= r - B)
        ring = []
        for rr in range(r - B + 1, r):
            ring += sorted(s for s in occ if self.last[s] == rr)
        return free + cold + ring

    def step(self, flat):
        self.round += 1
        uniq = list(dict.fromkeys(a for a in flat if a != synth.PAD))
        for a in uniq:
            if self.loc[a][0] == "G":
                self.last[self.loc[a][1]] = self.round
        misses = [a for a in uniq if self.loc[a][0] == "H"]
        hits = len(uniq) - len(misses)
        free_gpu = self.S - len(self.owner)
        free_host = self.H - len(self.host_owner)
        can_place = min(self.S - hits, free_gpu + free_host)
        if len(misses) > can_place:
            assert self.bypass, "capacity exceeded without the bypass"
            misses = misses[:can_place]  # the rest are read from the host pool in place
        victims = self.order()[:len(misses)]
        assert len(victims) == len(misses)
        owned = [v for v in victims if v in self.owner]
        host_free = sorted(h for h in range(self.H) if h not in self.host_owner)
        wb = host_free[:len(owned)]
        wbi = 0
        released = []
        for v, a in zip(victims, misses):
            if v in self.owner:
                o = self.owner[v]
                h = wb[wbi]
                wbi += 1
                self.host_owner[h], self.loc[o] = o, ("H", h)
            released.append(self.loc[a][1])
            self.owner[v], self.last[v], self.loc[a] = a, self.round, ("G", v)
        for h in released:
            del self.host_owner[h]
        return victims, wb


def _random_trace(rng, S, H, B, rounds, lru, n0, bypass=False, max_pick=None, exact=False):
    """Random tiny trace: selections with repeats and pads, allocs and frees between steps.
    exact: the oracle runs its exact-LRU mode (checked against lru=True)."""
    o = Oracle(ID_ROW_BYTES, [1], S, H, B, 4096, bypass=bypass, exact_lru=exact)
    bf = BruteForce(S, H, B, lru=lru, bypass=bypass)
    live = []
    assert o.alloc(n0, _id_row_buf(0, n0)) == bf.alloc(n0)
    live += list(range(n0))
    for _ in range(rounds):
        # between steps: occasionally free a live range or allocate a few
        if rng.random() < 0.15 and len(live) > S:
            a = rng.choice(live)
            o.free(a, 1)
            bf.free(a, 1)
            live.remove(a)
        if rng.random() < 0.2:
            n = rng.randint(1, 3)
            if len(live) + n + 8 <= S + H:
                base = bf.alloc(n)
                assert o.alloc(n, _id_row_buf(base, n)) == base
                live += list(range(base, base + n))
        k = rng.randint(1, max_pick if max_pick else min(S, 6))
        picks = rng.sample(live, min(k, len(live)))
        flat = []
        for a in picks:  # duplicates and pads inside the selection
            flat.append(a)
            if rng.random() < 0.3:
                flat.append(a)
            if rng.random() < 0.1:
                flat.append(synth.PAD)
        sel = np.array(flat, dtype=np.uint32).reshape(1, 1, -1)
        # the selection must fit next to the hits: M <= S - hits always holds when
        # the selection has at most S distinct addresses
        res = o.step_group(0, sel)
        v_bf, wb_bf = bf.step(flat)
        v, vc, wb = o.last_decisions(0)
        assert v.tolist() == v_bf
        assert wb.tolist() == wb_bf
        st = o.export(0)
        for a, (t, s) in bf.loc.items():
            assert st["tier"][a] == (TIER_GPU if t == "G" else TIER_HOST) and st["slot"][a] == s
        stamp, rounds_done = o.stamps(0)
        assert rounds_done == bf.round
        assert stamp.tolist() == [bf.last.get(x, 0xFFFFFFFF) for x in range(S)]
        got = res["out"][0, :res["req_off"][-1]].view(np.uint32)[:, 0]
        assert got.tolist() == list(dict.fromkeys(a for a in flat if a != synth.PAD))
    return o


@pytest.mark.parametrize("seed", range(60))
def test_no_fold_equals_round_lru(seed):
    """B > rounds: no bucket is ever reused, so PB-LRU is round-granular LRU."""
    rng = random.Random(seed)
    S = rng.randint(2, 16)
    rounds = rng.randint(5, 40)
    _random_trace(rng, S=S, H=64, B=rounds + 2, rounds=rounds, lru=True,
                  n0=rng.randint(S, S + 20))


@pytest.mark.parametrize("seed", range(120))
def test_with_folds_matches_timestamp_model(seed):
    rng = random.Random(1000 + seed)
    S = rng.randint(2, 16)
    B = rng.randint(2, 5)
    _random_trace(rng, S=S, H=64, B=B, rounds=rng.randint(10, 120), lru=False,
                  n0=rng.randint(S, S + 24))


@pytest.mark.parametrize("seed", range(80))
def test_overflow_bypass_matches_timestamp_model(seed):
    """Selections larger than the pool: the first S - hits misses become resident,
    the rest are gathered from the host pool in place (the gathered ids are checked
    inside _random_trace)."""
    rng = random.Random(5000 + seed)
    S = rng.randint(2, 10)
    B = rng.randint(2, 5)
    _random_trace(rng, S=S, H=rng.choice([16, 64]), B=B, rounds=rng.randint(10, 60), lru=False,
                  n0=rng.randint(S, S + 12), bypass=True, max_pick=2 * S + 3)


@pytest.mark.parametrize("seed", range(120))
def test_exact_lru_matches_timestamp_model(seed):
    """Exact LRU: free slots ascending, then occupied slots by (last round, slot),
    whatever the ring size (B is ignored by the policy)."""
    rng = random.Random(9000 + seed)
    S = rng.randint(2, 16)
    B = rng.randint(1, 5)
    _random_trace(rng, S=S, H=64, B=B, rounds=rng.randint(10, 120), lru=True,
                  n0=rng.randint(S, S + 24), exact=True)


@pytest.mark.parametrize("seed", range(40))
def test_exact_lru_bypass_matches_timestamp_model(seed):
    rng = random.Random(12000 + seed)
    S = rng.randint(2, 10)
    _random_trace(rng, S=S, H=rng.choice([16, 64]), B=rng.randint(1, 4), rounds=rng.randint(10, 60),
                  lru=True, n0=rng.randint(S, S + 12), bypass=True, max_pick=2 * S + 3, exact=True)


def test_overflow_without_bypass_is_an_error():
    o = Oracle(ID_ROW_BYTES, [1], 4, 16, 3, 64)
    o.alloc(10, _id_row_buf(0, 10))
    with pytest.raises(OracleError) as ei:
        o.step_group(0, np.arange(6, dtype=np.uint32).reshape(1, 1, 6))
    assert ei.value.code == CAPACITY
    ob = Oracle(ID_ROW_BYTES, [1], 4, 16, 3, 64, bypass=True)
    ob.alloc(10, _id_row_buf(0, 10))
    res = ob.step_group(0, np.arange(10, dtype=np.uint32).reshape(1, 1, 10))
    c = res["counters"]
    # slots 0..3 hold addresses 0..3 (hits); no slot is left for the 6 misses
    assert c["hits"] == 4 and c["misses"] == 6 and c["bypassed"] == 6
    got = res["out"][0, :10].view(np.uint32)[:, 0]
    assert got.tolist() == list(range(10))


def test_textbook_lru_differs_once_folds_happen():
    """Sanity of the pin above: the two brute-force orders are not the same policy."""
    differ = 0
    for seed in range(40):
        rng = random.Random(seed)
        S, B = 8, 2
        a, b = BruteForce(S, 64, B, lru=False), BruteForce(S, 64, B, lru=True)
        for m in (a, b):
            m.alloc(20)
        for _ in range(30):
            picks = rng.sample(range(20), 5)
            if a.step(picks)[0] != b.step(picks)[0]:
                differ += 1
                break
    assert differ > 0


# ----------------------------------------------------- workload-level pins

@pytest.mark.parametrize("name", ["tiny_1x4k", "batch8_32k", "longdoc", "low_evict", "low_overlap"])
def test_workload_closed_forms_and_invariants(name):
    w = WORKLOADS["tiny_1x4k"] if name == "tiny_1x4k" else small(name)
    w = w.replace(steps=min(w.steps, 24))
    run = OracleRun(w, mode="bytes")
    for t in range(w.steps):
        sel, ev, res = run.step()
        for g in range(w.n_groups):
            uniq = check_step_outputs(sel[g], res[g], g, w, "bytes")
            c = res[g]["counters"]
            assert c["uniq"] == len(uniq) and c["hits"] + c["misses"] == c["uniq"]
            assert c["victims_free"] + c["victims_cold"] + c["victims_ring"] == c["misses"]
            assert c["writebacks"] == c["misses"] - c["victims_free"]
        for g in range(w.n_groups):
            st = run.o.export(g)
            check_invariants(st, w.gpu_slots, w.host_slots, run.live)
            # the pools hold each address's own rows (moves copy whole slots intact)
            gp, hp = run.o.gpu_pool(g), run.o.host_pool(g)
            gpu_addrs = np.nonzero(st["tier"] == TIER_GPU)[0].astype(np.uint32)
            host_addrs = np.nonzero(st["tier"] == TIER_HOST)[0].astype(np.uint32)
            pick = np.random.default_rng(t).choice(gpu_addrs, min(64, len(gpu_addrs)), False)
            for j in range(w.layers_per_group):
                exp = synth.content_list(w.seed, g, j, pick, w.row_bytes)
                assert np.array_equal(gp[st["slot"][pick], j], exp)
            if len(host_addrs):
                pick = np.random.default_rng(t + 7).choice(host_addrs, min(64, len(host_addrs)),
                                                           False)
                exp = synth.content_list(w.seed, g, 0, pick, w.row_bytes)
                assert np.array_equal(hp[st["slot"][pick], 0], exp)


def test_current_round_never_evicted_and_all_selected_resident():
    w = small("low_overlap").replace(steps=16)
    run = OracleRun(w, mode="id")
    for _ in range(w.steps):
        sel_all, ev = run.trace.step()
        for g in range(w.n_groups):
            before = run.o.export(g)
            sel = sel_all[g]
            flat = sel.reshape(-1)
            flat = flat[flat != synth.PAD]
            hit_slots = {int(before["slot"][a]) for a in flat if before["tier"][a] == TIER_GPU}
            run.o.step_group(g, sel)
            v, vc, wb = run.o.last_decisions(g)
            assert not (set(v.tolist()) & hit_slots)
            after = run.o.export(g)
            assert (after["tier"][flat] == TIER_GPU).all()
            # hits stay where they were; every selected slot is in the current bucket
            for a in flat:
                if before["tier"][a] == TIER_GPU:
                    assert after["slot"][a] == before["slot"][a]
                assert after["cls"][after["slot"][a]] == after["cur"]
            # victims in class order: free, cold, then ring oldest -> newest
            rank = {FREE: 0, COLD: 1}
            B = w.ring_buckets
            keys = [rank.get(int(c), 2 + (int(c) - after["cur"] - 1) % B) for c in vc]
            assert keys == sorted(keys)
        from tests.harness import apply_events
        apply_events(run.alloc, run.free, ev)


def test_rotation_only_relabels():
    """A step whose selection is all hits moves no data and changes no map entry."""
    w = WORKLOADS["tiny_1x4k"]
    run = OracleRun(w, mode="bytes")
    st0 = run.o.export(0)
    gp0 = run.o.gpu_pool(0).copy()
    hp0 = run.o.host_pool(0).copy()
    resident = np.nonzero(st0["tier"] == TIER_GPU)[0][:200].astype(np.uint32)
    res = run.o.step_group(0, resident.reshape(1, 1, -1))
    assert res["counters"]["misses"] == 0
    st1 = run.o.export(0)
    assert np.array_equal(st0["tier"], st1["tier"]) and np.array_equal(st0["slot"], st1["slot"])
    assert np.array_equal(gp0, run.o.gpu_pool(0)) and np.array_equal(hp0, run.o.host_pool(0))
    assert st1["cur"] == (st0["cur"] + 1) % w.ring_buckets
    assert (st1["cls"][st1["slot"][resident]] == st1["cur"]).all()
    # everything else that was in the reused bucket is now cold
    others = np.setdiff1d(np.nonzero(st0["cls"] == st1["cur"])[0], st1["slot"][resident])
    assert (st1["cls"][others] == COLD).all()


def _state_equal(a, b):
    return all(np.array_equal(a[k], b[k]) for k in a)


def test_errors_leave_state_untouched():
    w = WORKLOADS["tiny_1x4k"]
    run = OracleRun(w, mode="bytes")
    for _ in range(3):
        run.step()
    st = run.o.export(0)
    gp = run.o.gpu_pool(0).copy()
    # unmapped: an address never allocated / out of range
    for bad in (w.max_logical - 1 if w.max_logical > 4096 else 5000, 0xFFFFFFF0):
        sel = np.array([1, 2, bad], dtype=np.uint32).reshape(1, 1, 3)
        with pytest.raises(OracleError) as ei:
            run.o.step_group(0, sel)
        assert ei.value.code == UNMAPPED
        assert _state_equal(st, run.o.export(0))
    # capacity: more distinct addresses than GPU slots
    host_addrs = np.nonzero(st["tier"] == TIER_HOST)[0]
    gpu_addrs = np.nonzero(st["tier"] == TIER_GPU)[0]
    sel = np.concatenate([gpu_addrs, host_addrs[:50]]).astype(np.uint32).reshape(1, 1, -1)
    with pytest.raises(OracleError) as ei:
        run.o.step_group(0, sel)
    assert ei.value.code == CAPACITY
    assert _state_equal(st, run.o.export(0))
    assert np.array_equal(gp, run.o.gpu_pool(0))
    # output buffer too small
    sel = gpu_addrs[:10].astype(np.uint32).reshape(1, 1, -1)
    with pytest.raises(OracleError) as ei:
        run.o.step_group(0, sel, out_cap=9)
    assert ei.value.code == CAPACITY
    assert _state_equal(st, run.o.export(0))
    # double free and out-of-range free
    run.o.free(10, 2)
    with pytest.raises(OracleError) as ei:
        run.o.free(11, 1)
    assert ei.value.code == INVALID_ARG
    with pytest.raises(OracleError) as ei:
        run.o.free(w.max_logical - 1, 2)
    assert ei.value.code == INVALID_ARG


def test_alloc_placement_and_free():
    o = Oracle(ID_ROW_BYTES, [2, 3], 5, 6, 4, 100)
    buf = np.concatenate([id_rows(0, 2, 0, 8).reshape(-1), id_rows(1, 3, 0, 8).reshape(-1)])
    assert o.alloc(8, buf) == 0
    for g in range(2):
        st = o.export(g)
        assert st["tier"][:5].tolist() == [TIER_GPU] * 5 and st["slot"][:5].tolist() == list(range(5))
        assert st["tier"][5:8].tolist() == [TIER_HOST] * 3 and st["slot"][5:8].tolist() == [0, 1, 2]
        assert (st["cls"] == st["cur"]).all()  # placed slots join the current bucket
    o.free(1, 2)     # GPU slots 1, 2 free
    o.free(6, 1)     # host slot 1 free
    buf = np.concatenate([id_rows(0, 2, 8, 4).reshape(-1), id_rows(1, 3, 8, 4).reshape(-1)])
    assert o.alloc(4, buf) == 8  # bases are never reused
    st = o.export(1)
    assert [st["slot"][a] for a in (8, 9)] == [1, 2] and st["tier"][8] == TIER_GPU
    assert [(st["tier"][a], st["slot"][a]) for a in (10, 11)] == [(TIER_HOST, 1), (TIER_HOST, 3)]
    with pytest.raises(OracleError) as ei:  # 9 live + 3 > S + H = 11
        o.alloc(3, np.concatenate([id_rows(0, 2, 12, 3).reshape(-1), id_rows(1, 3, 12, 3).reshape(-1)]))
    assert ei.value.code == CAPACITY
    # layer rows land in their own layer: gather of group 1 returns (g=1, j) tags
    res = o.step_group(1, np.array([[[8, 0]]], dtype=np.uint32))
    for j in range(3):
        ids = res["out"][j, :2].view(np.uint32)
        assert ids[:, 0].tolist() == [8, 0] and (ids[:, 1] == (1 << 16 | j)).all()


class _WithCompanion(OracleRun):
    """An oracle replay with the exact-LRU hit-rate companion stepped beside it."""

    def __init__(self, w):
        self.lru = ExactLru(w.n_groups, w.gpu_slots, w.max_logical)
        super().__init__(w, mode="id")

    def alloc(self, expect_base, n):
        assert self.lru.alloc(n) == expect_base
        return super().alloc(expect_base, n)

    def free(self, base, n):
        self.lru.free(base, n)
        super().free(base, n)

    def step(self):
        from tests.harness import apply_events
        sel, ev = self.trace.step()
        res = [self.o.step_group(g, sel[g]) for g in range(self.w.n_groups)]
        for g in range(self.w.n_groups):
            self.lru.step_group(g, sel[g])
        apply_events(self.alloc, self.free, ev)
        return sel, ev, res


@pytest.mark.parametrize("name", ["batch8_32k", "low_overlap"])
def test_exact_lru_companion_agrees_with_exact_mode(name):
    """The hit-rate companion and the oracle's exact-LRU mode are the same policy:
    same hits and unique rows on the same trace (turnover included)."""
    w = small(name).replace(steps=20, exact_lru=True)
    run = _WithCompanion(w)
    uniq = hits = 0
    for _ in range(w.steps):
        sel, ev, res = run.step()
        for g in range(w.n_groups):
            uniq += res[g]["counters"]["uniq"]
            hits += res[g]["counters"]["hits"]
    assert int(run.lru.acc[0]) == uniq and int(run.lru.acc[1]) == hits
    assert 0 < hits < uniq


def test_exact_lru_companion_sanity():
    """Parity unpinned (reported only); sanity: a pool larger than the history only
    misses never, and a cold start with a tiny pool misses."""
    lru = ExactLru(1, 4096, 1000)
    lru.alloc(1000)
    rng = np.random.default_rng(0)
    for _ in range(10):
        lru.step_group(0, rng.choice(1000, 50, replace=False).astype(np.uint32))
    assert lru.hit_rate == 1.0
    lru2 = ExactLru(1, 8, 1000)
    lru2.alloc(1000)
    for _ in range(10):
        lru2.step_group(0, rng.choice(1000, 8, replace=False).astype(np.uint32))
    assert lru2.hit_rate < 0.5
