"""Pins of the TP-mode emulation in the oracle (UlaCache summary page, §2 TP
paragraph): striping t -> partition t mod P, each partition a DP residency over
its own addresses; per rank and group a local buffer of remote rows.

* closed forms: every local output row is the generator's row of an owned selected
  address, every remote output row that of a non-owned one, each in first-occurrence
  order; every buffered slot holds the row of the address it maps;
* a brute-force model of the buffer written with per-slot timestamps (PB-LRU order:
  free ascending, cold = last access at least B rounds old, ascending, then the ring
  rounds oldest to newest; a victim's copy dropped), on random tiny traces;
* with P = 1 the partition is exactly the DP oracle on the same trace;
* invariants: every remote selected address is buffered after the step, buffer map
  and owners agree, never-both holds in every partition.
"""
from __future__ import annotations

import random

import numpy as np
import pytest

import synth
from oracle import COLD, FREE, Oracle, OracleTP
from tests.harness import ID_ROW_BYTES, check_invariants, id_rows


def _rows(n, base, layers):
    return np.concatenate([id_rows(g, L, base, n).reshape(-1) for g, L in enumerate(layers)])


def _ids(out, U):
    return out[:, :U].view(np.uint32).reshape(out.shape[0], U, 2)


class BufferBruteForce:
    def __init__(self, slots, B):
        self.slots, self.B = slots, B
        self.addr = {}   # slot -> address
        self.last = {}   # slot -> last round
        self.where = {}  # address -> slot
        self.round = 0

    def drop(self, a):
        s = self.where.pop(a, None)
        if s is not None:
            del self.addr[s], self.last[s]

    def order(self):
        free = [s for s in range(self.slots) if s not in self.addr]
        occ = [s for s in self.addr if self.last[s] != self.round]
        r, B = self.round, self.B
        cold = sorted(s for s in occ if self.last[s] <= r - B)
        ring = []
        for rr in range(r - B + 1, r):
            ring += sorted(s for s in occ if self.last[s] == rr)
        return free + cold + ring

    def step(self, remote_uniq):
        self.round += 1
        for a in remote_uniq:
            if a in self.where:
                self.last[self.where[a]] = self.round
        misses = [a for a in remote_uniq if a not in self.where]
        victims = self.order()[:len(misses)]
        assert len(victims) == len(misses)
        for v, a in zip(victims, misses):
            if v in self.addr:
                del self.where[self.addr[v]]
            self.addr[v], self.last[v], self.where[a] = a, self.round, v
        return victims


def _check_step(o, res, sel_g, g, P, layers):
    flat = sel_g.reshape(-1)
    valid = flat[flat != synth.PAD]
    for r in range(P):
        own = [int(a) for a in dict.fromkeys(valid.tolist()) if a % P == r]
        rem = [int(a) for a in dict.fromkeys(valid.tolist()) if a % P != r]
        loc, rmt = res[r]["local"], res[r]["remote"]
        Ul, Ur = int(loc["req_off"][-1]), int(rmt["req_off"][-1])
        assert (Ul, Ur) == (len(own), len(rem))
        li, ri = _ids(loc["out"], Ul), _ids(rmt["out"], Ur)
        for j in range(layers[g]):
            assert li[j, :, 0].tolist() == own and (li[j, :, 1] == (g << 16 | j)).all()
            assert ri[j, :, 0].tolist() == rem and (ri[j, :, 1] == (g << 16 | j)).all()
        # entry rows point at their address's row, -1 for the other side and pads
        er = rmt["entry_row"]
        for e, a in enumerate(flat.tolist()):
            if a == synth.PAD or a % P == r:
                assert er[e] == -1
            else:
                assert rem[er[e]] == a
        # every remote selected address is buffered, and the buffer holds its row
        buf = o.buffer(r, g)
        where, owner = buf["where"], buf["owner"]
        for a in rem:
            assert where[a] >= 0 and owner[where[a]] == a
        held = np.nonzero(where >= 0)[0]
        assert len(np.unique(where[held])) == len(held)
        assert (owner[where[held]] == held).all()
        assert ((buf["cls"] == FREE) == (owner == 0xFFFFFFFF)).all()


def _trace(rng, P, S, H, B, slots, rounds, layers=(1,), n0=None, max_pick=None):
    max_logical = 4096
    o = OracleTP(ID_ROW_BYTES, list(layers), P, S, H, B, max_logical, slots)
    bf = [[BufferBruteForce(slots, B) for _ in layers] for _ in range(P)]
    n0 = n0 if n0 is not None else P * S + rng.randint(0, 8)
    assert o.alloc(n0, _rows(n0, 0, layers)) == 0
    live = list(range(n0))
    nxt = n0
    for _ in range(rounds):
        if rng.random() < 0.2:  # appends
            n = rng.randint(1, 3)
            assert o.alloc(n, _rows(n, nxt, layers)) == nxt
            live += list(range(nxt, nxt + n))
            nxt += n
        g = rng.randrange(len(layers))
        # at most S distinct owned addresses per partition, `slots` remote ones per rank
        k = rng.randint(1, max_pick or min(S, slots))
        picks = rng.sample(live, min(k, len(live)))
        flat = []
        for a in picks:
            flat.append(a)
            if rng.random() < 0.3:
                flat.append(a)
            if rng.random() < 0.1:
                flat.append(synth.PAD)
        sel = np.array(flat, dtype=np.uint32).reshape(1, 1, -1)
        res = o.step_group(g, sel)
        _check_step(o, res, sel, g, P, list(layers))
        uniq = list(dict.fromkeys(a for a in flat if a != synth.PAD))
        for r in range(P):
            v = bf[r][g].step([a for a in uniq if a % P != r])
            assert o.buffer(r, g)["victims"].tolist() == v, (r, g)
        for p in range(P):
            st = o.partition(p).export(g)
            live_p = {a // P for a in live if a % P == p}
            check_invariants(st, S, H, live_p)
    return o


@pytest.mark.parametrize("seed", range(60))
def test_tp_buffer_matches_timestamp_model(seed):
    rng = random.Random(20000 + seed)
    P = rng.choice([2, 3, 4])
    S = rng.randint(3, 10)
    slots = rng.randint(2, 3 * S)
    _trace(rng, P, S, H=64, B=rng.randint(2, 5), slots=slots, rounds=rng.randint(10, 60),
           layers=rng.choice([(1,), (2, 1)]))


def test_tp_one_partition_is_the_dp_oracle():
    rng = random.Random(7)
    layers = (2,)
    S, H, B = 6, 64, 3
    tp = OracleTP(ID_ROW_BYTES, list(layers), 1, S, H, B, 4096, 4)
    dp = Oracle(ID_ROW_BYTES, list(layers), S, H, B, 4096)
    n0 = 30
    assert tp.alloc(n0, _rows(n0, 0, layers)) == 0 and dp.alloc(n0, _rows(n0, 0, layers)) == 0
    for _ in range(40):
        sel = np.array(rng.sample(range(n0), 5), dtype=np.uint32).reshape(1, 1, -1)
        a = tp.step_group(0, sel)[0]
        b = dp.step_group(0, sel)
        assert np.array_equal(a["local"]["out"], b["out"])
        assert np.array_equal(a["local"]["entry_row"], b["entry_row"])
        assert a["remote"]["req_off"][-1] == 0 and (a["remote"]["entry_row"] == -1).all()
        sa, sb = tp.partition(0).export(0), dp.export(0)
        assert all(np.array_equal(sa[k], sb[k]) for k in sa)


def test_tp_buffer_hit_rate_follows_overlap():
    """Consecutive selections that overlap heavily keep the remote rows buffered (the
    pages' reason for the buffer); selections of never-seen addresses fetch every
    remote row."""
    P, S, slots = 4, 512, 256
    for overlap, lo, hi in ((0.9, 0.85, 0.95), (0.0, 0.0, 0.0)):
        o = OracleTP(ID_ROW_BYTES, [1], P, S, 1024, 4, 8192, slots)
        n0 = 4000
        o.alloc(n0, _rows(n0, 0, (1,)))
        nxt = 0  # addresses are drawn fresh from here on
        prev = np.arange(100, dtype=np.uint32)
        nxt = 100
        hits = tot = 0
        for t in range(30):
            keep = prev[: int(overlap * len(prev))]
            fresh = np.arange(nxt, nxt + 100 - len(keep), dtype=np.uint32)
            nxt += len(fresh)
            cur = np.concatenate([keep, fresh]).astype(np.uint32)
            res = o.step_group(0, cur.reshape(1, 1, -1))
            if t >= 1:
                for r in range(P):
                    hits += res[r]["remote"]["counters"]["hits"]
                    tot += res[r]["remote"]["counters"]["uniq"]
            prev = cur
        assert lo <= hits / tot <= hi, (overlap, hits / tot)
