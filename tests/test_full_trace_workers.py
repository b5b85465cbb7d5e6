"""The whole-trace replay's oracle processes (CPU): spawned per-group workers send, step by
step, the same unique addresses, offsets, entry-row digests and state digests as the
multi-group oracle run in this process on the same trace."""
from __future__ import annotations

import numpy as np

from oracle.replay import OracleRun
from synth.configs import WORKLOADS
from tests.full_trace import OracleWorkers, digest, state_digests

OVERRIDES = dict(n_live=4, ctx_min=3000, ctx_max=6000, k=256, window=64, steps=7, append_cap=64)


def test_workers_match_the_oracle_in_process():
    w = WORKLOADS["longdoc"].replace(**OVERRIDES)
    workers = OracleWorkers("longdoc", OVERRIDES, w.n_groups, w.steps, state_every=3)
    try:
        run = OracleRun(w, "id")
        for g in range(w.n_groups):
            workers.recv(g, "ready", timeout=120)
        for t in range(w.steps):
            sel, ev = run.trace.step()
            for g in range(w.n_groups):
                res = run.o.step_group(g, sel[g])
                msg = workers.recv(g, "step", timeout=120)
                U = int(res["req_off"][-1])
                assert msg["t"] == t and msg["U"] == U
                assert np.array_equal(msg["req_off"], res["req_off"])
                assert msg["entry_row"] == digest(res["entry_row"])
                ids = res["out"][0, :U].view(np.uint32).reshape(U, 2)
                assert np.array_equal(msg["uniq"], ids[:, 0])
                if (t + 1) % 3 == 0 or t == w.steps - 1:
                    st = dict(run.o.export(g))
                    st["stamp"] = run.o.stamps(g)[0]
                    v, _vc, wb = run.o.last_decisions(g)
                    assert msg["state"] == state_digests(st, (v, wb))
                else:
                    assert "state" not in msg
            for kind in ("free", "join", "append"):
                if ev[f"{kind}_n"]:
                    if kind == "free":
                        run.free(ev["free_base"], ev["free_n"])
                    else:
                        run.alloc(ev[f"{kind}_base"], ev[f"{kind}_n"])
        for g in range(w.n_groups):
            workers.recv(g, "done", timeout=120)
    finally:
        workers.close()


def test_digest_is_elementwise():
    a = np.arange(10, dtype=np.uint32)
    b = a.copy()
    assert digest(a) == digest(b) == digest(a.astype(np.int64))
    b[7] ^= 1
    assert digest(a) != digest(b)
