"""Replica aggregation of the benchmark (N > 1): world_size-2 gloo ranks on CPU.

The path has no exchange step (DP ranks are independent replicas), so the only
collectives are the timing barrier and the MAX-of-times / SUM-of-work reduction
that turns per-rank results into the whole-job value.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, l = bench.dist_env()
    assert (r, w, l) == (rank, world, rank)
    dist.barrier()
    out = bench.aggregate({"rows": 1000.0 * (rank + 1), "value_ms": 10.0 + 5 * rank,
                           "e2e_ms": 3.0 - rank}, world, torch.device("cpu"))
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replica_aggregation_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert res[r]["rows"] == 3000.0          # SUM of work over replicas
        assert res[r]["value_ms"] == 15.0        # the slowest rank's time
        assert res[r]["e2e_ms"] == 3.0
    # whole-job value = all ranks' rows / the slowest time
    assert res[0]["rows"] / (res[0]["value_ms"] / 1e3) == pytest.approx(200000.0)


def test_single_rank_aggregation_is_identity():
    import bench
    assert bench.aggregate({"rows": 5.0, "value_ms": 2.0}, 1) == {"rows": 5.0, "value_ms": 2.0}


def test_reference_arm_line(capsys):
    """`bench.py --impl reference` prints one JSON line with the contract's keys: the oracle
    timed single-threaded on a bounded sample, its e2e equal to its value, no host copies."""
    import json

    import bench
    assert bench.main(["--impl", "reference", "--workload", "tiny_1x4k", "--steps", "4",
                       "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "rows/s" and line["value"] > 0
    assert line["steps"] == 4 and line["warmup"] == 3 and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("1 request")


def test_roofline_helpers(monkeypatch):
    """The gather's DRAM traffic per launch: the two launch kinds' per-row figures times
    the hits, averaged over launches; withheld once the kernel's source hash moves."""
    import bench
    t = dict(bench.GATHER_TRAFFIC)
    # DRAM reads cover at least the algorithmic reads: one 656-byte row, three of a slot
    assert 656 <= t["layer0_bytes_per_row"] < 2 * 656
    assert 3 * 656 <= t["later_bytes_per_slot"] < 2 * 3 * 656
    monkeypatch.setattr(bench, "gather_source_sha256", lambda: t["source_sha256"])
    hits, L, launches = 1000, 4, 2
    exp = hits * (t["layer0_bytes_per_row"] + t["later_bytes_per_slot"]) / launches
    assert bench.traffic_per_launch(hits, L, launches) == round(exp)
    assert bench.traffic_per_launch(hits, 1, 1) == round(hits * t["layer0_bytes_per_row"])
    assert bench.traffic_per_launch(hits, L, 0) is None
    monkeypatch.setattr(bench, "gather_source_sha256", lambda: "0" * 64)
    assert bench.traffic_per_launch(hits, L, launches) is None
    peak, src = bench.measured_peaks()
    assert peak > 1000 and src in ("measured", "fallback")
