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
    assert cb["host_cores"] == os.cpu_count() and cb["pinned_core"] in os.sched_getaffinity(0)
    assert os.sched_getaffinity(0) != {cb["pinned_core"]} or os.cpu_count() == 1  # restored
    assert line["e2e"] == {"value": line["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("1 request")


def test_roofline_helpers(monkeypatch):
    """Span bookkeeping (union of overlapping launch spans, per-kernel sums) and the
    gather's DRAM traffic per launch from the ncu figures per hit row, withheld once the
    kernel's source hash moves or on another workload."""
    import bench
    assert bench.union_ns([]) == 0
    assert bench.union_ns([(0, 10), (5, 20), (30, 40)]) == 30
    assert bench.union_ns([(30, 40), (0, 10), (10, 12)]) == 22
    spans = [("gather", 0, 100, 300), ("move", 0, 300, 1300), ("gather", 1, 1300, 1500),
             ("move", 1, 1500, 2500), ("stage", 1, 0, 0)]  # an empty record is skipped
    sm = bench.span_summary(spans, {}, 4, 656, 2)
    assert sm["gather"] == {"launches": 2, "sum_us": 0.4, "union_us": 0.4}
    assert bench.overlap_ns([(0, 10), (20, 30)], [(5, 25)]) == 10
    assert bench.overlap_ns([(0, 10)], [(10, 20)]) == 0
    spans2 = spans + [("select", 1, 200, 1400)]  # metadata beside the move and the gather
    assert bench.span_summary(spans2, {}, 4, 656, 2)["select"]["beside_copies_us"] == 1.2
    assert sm["move"]["launches"] == 2 and sm["move"]["sum_us"] == 2.0 and "stage" not in sm
    t = dict(bench.GATHER_TRAFFIC)
    if t["source_sha256"] is not None:  # DRAM reads cover at least the algorithmic reads
        assert 4 * 656 <= t["read_bytes_per_hit"] < 2 * 4 * 656
        assert t["hit_rows"] > 0 and t["workload"]
    fake = {"source_sha256": "f" * 64, "workload": "longdoc", "hit_rows": 100,
            "read_bytes_per_hit": 2700.0, "write_bytes_per_hit": 2624.0}
    monkeypatch.setattr(bench, "GATHER_TRAFFIC", fake)
    monkeypatch.setattr(bench, "gather_source_sha256", lambda: "f" * 64)
    assert bench.traffic_per_launch(1000, 2, "longdoc") == round(1000 * (2700 + 2624) / 2)
    assert bench.traffic_per_launch(1000, 0, "longdoc") is None
    assert bench.traffic_per_launch(1000, 2, "low_evict") is None
    monkeypatch.setattr(bench, "gather_source_sha256", lambda: "0" * 64)
    assert bench.traffic_per_launch(1000, 2, "longdoc") is None
    peak, src = bench.measured_peaks()
    assert peak > 1000 and src in ("measured", "fallback")
