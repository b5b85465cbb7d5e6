"""The five synthetic workloads of the KV residency path, and small variants for tests.

Each workload is a decode trace: requests with long histories of logical KV
addresses, G selection groups (each group of L_g layers shares one top-k
selection, UlaCache page "Unified logical addresses", the two extra details),
a GPU slot pool sized as a fraction of the history (the rest lives in pinned
host memory; an entry is in exactly one of the two) and a per-step
selection with a recent window, a kept fraction of the previous selection
and fresh positions (uniform, or Zipf over position for the low-overlap
stress case).

Pool sizing: S (GPU slots per group) = floor(gpu_frac * total history)
unless given; H (host slots per group) = largest live history - S + one
step's worth of entries (R*Q*k), which is the write-back headroom an
exclusive two-tier pool needs: every victim that holds data takes a free
host slot before the misses' host slots are released.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    description: str
    seed: int
    n_live: int                 # R: requests decoding at once
    ctx_min: int                # initial context, uniform integer in [ctx_min, ctx_max]
    ctx_max: int
    n_groups: int               # G selection groups
    layers_per_group: int       # L_g
    q: int                      # query tokens per request per step (unioned, deduped)
    k: int                      # top-k per query token
    window: int                 # recent window, always selected
    keep: float                 # fraction of the non-window budget kept from the previous set
    steps: int                  # decode steps of the trace
    fresh: str = "uniform"      # "uniform" | "zipf"
    zipf_s: float = 1.1
    n_total: int | None = None  # requests over the trace (turnover); default n_live
    append_max: int = 0         # accepted tokens appended per request per step, uniform [1, max]
    append_cap: int = 0         # cap on appended tokens per request
    turnover_period: int = 0    # every P steps the oldest request finishes and the next joins
    gpu_frac: float | None = None
    gpu_slots_explicit: int | None = None
    host_slots_explicit: int | None = None
    ring_buckets: int = 8       # B ring buckets (+ one cold bucket)
    row_bytes: int = 656        # 512 e4m3 latent + 4 fp32 scales + 64 bf16 rope
    pad_prob: float = 0.0       # fraction of entries replaced by the pad marker (edge tests)
    bypass: bool = False        # overflow bypass: misses beyond the pool are read in place
    exact_lru: bool = False     # exact LRU (timestamp per slot) in place of PB-LRU
    layer_signal: bool = False  # layer-major fill with a device flag per layer
    gather_beside: bool = False  # the hit gather runs beside the move (not before it)
    _cache: dict = field(default_factory=dict, compare=False, hash=False, repr=False)

    @property
    def total_requests(self) -> int:
        return self.n_total if self.n_total is not None else self.n_live

    def ctx_of(self, rid: int) -> int:
        from . import request_ctx
        return request_ctx(self, rid)

    def _ctxs(self):
        if "ctx" not in self._cache:
            if self.ctx_min == self.ctx_max:
                self._cache["ctx"] = [self.ctx_min] * self.total_requests
            else:
                self._cache["ctx"] = [self.ctx_of(i) for i in range(self.total_requests)]
        return self._cache["ctx"]

    @property
    def history_total(self) -> int:
        return sum(self._ctxs())

    @property
    def max_live_history(self) -> int:
        c = self._ctxs()
        best = max(sum(c[i:i + self.n_live]) for i in range(self.total_requests - self.n_live + 1))
        return best + (self.n_live * self.append_cap if self.append_max else 0)

    @property
    def entries_per_step(self) -> int:
        return self.n_live * self.q * self.k

    @property
    def gpu_slots(self) -> int:
        if self.gpu_slots_explicit is not None:
            return self.gpu_slots_explicit
        return int(math.floor(self.gpu_frac * self.history_total))

    @property
    def host_slots(self) -> int:
        if self.host_slots_explicit is not None:
            return self.host_slots_explicit
        return max(0, self.max_live_history - self.gpu_slots + self.entries_per_step)

    @property
    def max_logical(self) -> int:
        return self.history_total + (self.n_live * self.append_cap if self.append_max else 0)

    def replace(self, **kw) -> "Workload":
        kw.setdefault("_cache", {})
        return dataclasses.replace(self, **kw)

    def summary(self) -> dict:
        return {"workload": self.description, "requests": self.total_requests,
                "live_requests": self.n_live, "groups": self.n_groups,
                "layers_per_group": self.layers_per_group, "top_k": self.k,
                "query_tokens": self.q, "gpu_slots": self.gpu_slots,
                "host_slots": self.host_slots, "ring_buckets": self.ring_buckets,
                "row_bytes": self.row_bytes, "trace_steps": self.steps, "seed": self.seed,
                "policy": "exact LRU" if self.exact_lru else "PB-LRU"}


WORKLOADS = {
    "tiny_1x4k": Workload(
        name="tiny_1x4k", seed=0,
        description="1 request x 4,096 ctx, 1 group x 4 layers, top-256, GPU pool 2,048 slots",
        n_live=1, ctx_min=4096, ctx_max=4096, n_groups=1, layers_per_group=4, q=1, k=256,
        window=64, keep=0.85, steps=64, gpu_slots_explicit=2048, host_slots_explicit=4096),
    "batch8_32k": Workload(
        name="batch8_32k", seed=1,
        description="8 requests x 32K ctx, 4 groups x 3 layers, top-2,048, GPU pool 40% of history",
        n_live=8, ctx_min=32768, ctx_max=32768, n_groups=4, layers_per_group=3, q=1, k=2048,
        window=512, keep=0.9, steps=256, gpu_frac=0.4),
    "longdoc": Workload(
        name="longdoc", seed=2,
        description=("long-document summary: 32 requests x 64K-128K ctx (+<=1,024 appended), "
                     "4 groups x 4 layers, top-2,048 x 3 query tokens, GPU pool 30% of history"),
        n_live=32, ctx_min=65536, ctx_max=131072, n_groups=4, layers_per_group=4, q=3, k=2048,
        window=512, keep=0.9, steps=512, append_max=3, append_cap=1024, gpu_frac=0.3),
    "low_evict": Workload(
        name="low_evict", seed=3,
        description="low eviction: 16 requests x 64K ctx, 4 groups x 4 layers, top-2,048, GPU pool 95%",
        n_live=16, ctx_min=65536, ctx_max=65536, n_groups=4, layers_per_group=4, q=1, k=2048,
        window=512, keep=0.95, steps=512, gpu_frac=0.95),
    "low_overlap": Workload(
        name="low_overlap", seed=4,
        description=("low overlap: 256 requests x 16K ctx (192 live, turnover every 4 steps), "
                     "2 groups x 4 layers, top-2,048, overlap 0.5 + Zipf(1.1), GPU pool 10%"),
        n_live=192, n_total=256, ctx_min=16384, ctx_max=16384, n_groups=2, layers_per_group=4,
        q=1, k=2048, window=512, keep=0.5, fresh="zipf", zipf_s=1.1, steps=256,
        turnover_period=4, gpu_frac=0.1),
    # The low-overlap stress as literally stated: all 256 requests at once.  One step
    # selects 524,288 rows against 419,430 GPU slots, so it needs the overflow bypass.
    "low_overlap_256": Workload(
        name="low_overlap_256", seed=4,
        description=("low overlap, literal: 256 requests x 16K ctx all at once, 2 groups x 4 "
                     "layers, top-2,048, overlap 0.5 + Zipf(1.1), GPU pool 10%, overflow bypass"),
        n_live=256, ctx_min=16384, ctx_max=16384, n_groups=2, layers_per_group=4,
        q=1, k=2048, window=512, keep=0.5, fresh="zipf", zipf_s=1.1, steps=256,
        gpu_frac=0.1, bypass=True),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


def small(name: str, **kw) -> Workload:
    """A reduced copy of a workload (same recipe, smaller sizes) for full-state parity tests."""
    w = WORKLOADS[name]
    shrink = {
        "tiny_1x4k": dict(),
        "batch8_32k": dict(n_live=4, ctx_min=4096, ctx_max=4096, k=256, window=64, steps=48),
        "longdoc": dict(n_live=6, ctx_min=3000, ctx_max=6000, k=256, window=64, steps=40,
                     append_cap=64),
        "low_evict": dict(n_live=4, ctx_min=4096, ctx_max=4096, k=256, window=64, steps=48),
        "low_overlap": dict(n_live=12, n_total=20, ctx_min=2048, ctx_max=2048, k=256, window=64,
                     steps=40, turnover_period=4),
        "low_overlap_256": dict(n_live=20, ctx_min=2048, ctx_max=2048, k=256, window=64, steps=40),
    }[name]
    shrink.update(kw)
    return w.replace(name=name + "_small", description=w.description + " (reduced)", **shrink)
