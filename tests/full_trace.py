"""Whole-trace replay at full size: the GPU path against the oracle over every step of a
workload's trace.

The oracle runs in id mode (8-byte rows that name their address, group and layer; exact,
since a row's bytes are a function of those) in one child process per group (the groups
are independent: each has its own map, pools and ring, and alloc/free apply to each
alike), started with `spawn`.  A child replays the whole trace -- its group's steps and
every step's joins, finishes and appended tokens -- and sends per step what the GPU side
compares: the unique addresses in order (`uniq`), the CSR offsets, a digest of the entry
rows, and on state steps digests of the full state (map tiers and slots, class of every
GPU slot, slot owners, host-free set, host-slot owners, slot timestamps, the step's
victims and write-back slots).  Digests are SHA-256 of the arrays as int64, so equal
digests mean equal arrays element by element.
"""
from __future__ import annotations

import hashlib
import multiprocessing as mp

import numpy as np

STATE_KEYS = ("tier", "slot", "cls", "owner", "host_free", "host_owner", "stamp")


def digest(a) -> str:
    return hashlib.sha256(np.ascontiguousarray(np.asarray(a), dtype=np.int64).tobytes()).hexdigest()


def state_digests(st: dict, decisions) -> dict:
    d = {k: digest(st[k]) for k in STATE_KEYS}
    d["cur"] = int(st["cur"])
    v, wb = decisions
    d["victims"] = digest(v)
    d["wb_host"] = digest(wb)
    d["M"], d["K"] = int(len(v)), int(len(wb))
    return d


def oracle_worker(name: str, overrides: dict, g: int, steps: int, state_every: int, conn):
    """Child process: group g's oracle over the first `steps` steps of the workload."""
    import os
    os.environ.setdefault("OMP_NUM_THREADS", "2")  # (the trace generator; one child per group)
    from oracle.replay import OracleRun
    from synth.configs import WORKLOADS
    try:
        w = WORKLOADS[name].replace(**overrides) if overrides else WORKLOADS[name]
        run = OracleRun(w, "id")
        o = run.o
        L = w.layers_per_group
        conn.send(("ready", None))
        for t in range(steps):
            sel, ev = run.trace.step()
            res = o.step_group(g, sel[g])
            U = int(res["req_off"][-1])
            ids = res["out"][:, :U].view(np.uint32).reshape(L, U, 2)
            uniq = ids[0, :, 0].copy()
            for j in range(L):  # every layer's row names the same address, this group, layer j
                assert np.array_equal(ids[j, :, 0], uniq) and (ids[j, :, 1] == ((g << 16) | j)).all()
            msg = {"t": t, "U": U, "req_off": res["req_off"].copy(),
                   "entry_row": digest(res["entry_row"]), "uniq": uniq,
                   "counters": res["counters"]}
            if (t + 1) % state_every == 0 or t == steps - 1:
                st = dict(o.export(g))
                st["stamp"] = o.stamps(g)[0]
                v, _vc, wb = o.last_decisions(g)
                msg["state"] = state_digests(st, (v, wb))
            # the step's events, in the order the generator assigned logical ranges
            if ev["free_n"]:
                run.free(ev["free_base"], ev["free_n"])
            if ev["join_n"]:
                run.alloc(ev["join_base"], ev["join_n"])
            if ev["append_n"]:
                run.alloc(ev["append_base"], ev["append_n"])
            conn.send(("step", msg))
        conn.send(("done", None))
    except Exception as e:  # reported to the parent, which fails the test
        conn.send(("error", repr(e)))
    finally:
        conn.close()


class OracleWorkers:
    """One spawned oracle process per group, each sending per-step messages."""

    def __init__(self, name: str, overrides: dict, n_groups: int, steps: int, state_every: int):
        ctx = mp.get_context("spawn")
        self.procs, self.conns = [], []
        for g in range(n_groups):
            a, b = ctx.Pipe(duplex=False)
            p = ctx.Process(target=oracle_worker, args=(name, overrides, g, steps, state_every, b),
                            daemon=True)
            p.start()
            b.close()
            self.procs.append(p)
            self.conns.append(a)

    def recv(self, g: int, kind: str, timeout: float = 900.0):
        if not self.conns[g].poll(timeout):
            raise TimeoutError(f"oracle worker {g}: no message within {timeout} s")
        k, payload = self.conns[g].recv()
        if k == "error":
            raise RuntimeError(f"oracle worker {g}: {payload}")
        assert k == kind, (k, kind)
        return payload

    def close(self):
        for c in self.conns:
            c.close()
        for p in self.procs:
            p.join(timeout=5)
            if p.is_alive():
                p.terminate()
                p.join(timeout=5)
