"""GPU-side test driver: replays a workload through the CUDA library (C ABI via
the ctypes binding) and compares its state and outputs with the oracle's."""
from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import COLD, FREE, TIER_GPU, TIER_HOST, TIER_UNALLOCATED
from serving_step_sparse_gb300 import ula
from serving_step_sparse_gb300.cache import UlaCache
from tests.harness import ID_ROW_BYTES, apply_events, initial_allocs

STAGE_ADDRS = 16384  # addresses per staged alloc chunk


class GpuReplay:
    """group_streams: each group's call on a caller stream of its own (as the benchmark
    issues them: later groups' steps run ahead of earlier groups' copies)."""

    def __init__(self, w, out_cap: int | None = None, stage_addrs: int = STAGE_ADDRS,
                 group_streams: bool = False):
        self.w = w
        G, L = w.n_groups, w.layers_per_group
        self.cache = UlaCache(row_bytes=w.row_bytes, layers_per_group=[L] * G,
                              gpu_slots=w.gpu_slots, host_slots=w.host_slots,
                              ring_buckets=w.ring_buckets, max_logical=w.max_logical,
                              max_entries=w.entries_per_step, bypass_overflow=w.bypass,
                              exact_lru=w.exact_lru, layer_signal=w.layer_signal,
                              gather_beside_move=w.gather_beside)
        self.cap = out_cap if out_cap is not None else w.entries_per_step
        self.outs = [self.cache.out_buffer(g, self.cap) for g in range(G)]
        E = w.entries_per_step
        dev = self.cache.device
        self.entry_row = [torch.empty(E, dtype=torch.int32, device=dev) for _ in range(G)]
        self.req_off = [torch.empty(w.n_live + 1, dtype=torch.int32, device=dev) for _ in range(G)]
        self.sel_d = torch.empty((G, w.n_live, w.q, w.k), dtype=torch.int32, device=dev)
        self.stage_addrs = stage_addrs
        self.stage = torch.empty(stage_addrs * G * L * w.row_bytes, dtype=torch.uint8,
                                 pin_memory=True)
        self.trace = synth.Trace(w)
        self.live = set()
        self.gstreams = [torch.cuda.Stream(dev) for _ in range(G)] if group_streams else None
        for base, n in initial_allocs(w, self.trace):
            self.alloc(base, n)

    def close(self):
        self.cache.close()

    def alloc(self, expect_base, n):
        w = self.w
        G, L, W = w.n_groups, w.layers_per_group, w.row_bytes
        off = 0
        while off < n:
            m = min(self.stage_addrs, n - off)
            buf = self.stage[: m * G * L * W]
            view = buf.numpy().reshape(G, m, L, W)
            for g in range(G):
                synth.content_range(w.seed, g, L, expect_base + off, m, W, out=view[g])
            got = self.cache.alloc(m, buf)
            assert got == expect_base + off, (got, expect_base + off)
            self.cache.sync()  # the staging buffer is reused
            off += m
        self.live.update(range(expect_base, expect_base + n))
        return expect_base

    def free(self, base, n):
        self.cache.free(base, n)
        self.live.difference_update(range(base, base + n))

    def run_groups(self, sel: np.ndarray):
        self.sel_d.copy_(torch.from_numpy(np.ascontiguousarray(sel).view(np.int32)))
        main = self.cache.stream
        for g in range(self.w.n_groups):
            s = None
            if self.gstreams:
                s = self.gstreams[g]
                s.wait_stream(main)
            self.cache.step_group(g, self.sel_d[g], self.outs[g], self.entry_row[g],
                                  self.req_off[g], stream=s)
        if self.gstreams:
            for s in self.gstreams:
                main.wait_stream(s)
        return self.cache.sync()

    def step(self):
        sel, ev = self.trace.step()
        stats = self.run_groups(sel)
        apply_events(self.alloc, self.free, ev)
        return sel, ev, stats

    def results(self, g: int, full_out: bool = True):
        req_off = self.req_off[g].cpu().numpy()
        U = int(req_off[-1])
        res = {"req_off": req_off, "entry_row": self.entry_row[g].cpu().numpy()}
        if full_out:
            res["out"] = self.outs[g][:, :U].cpu().numpy()
        return res


class _DeviceWords:
    """A device array the library owns, seen through the CUDA array interface."""

    def __init__(self, ptr: int, n: int):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (ptr, False),
                                         "version": 2}


def check_layer_signal(cache, g: int, layers: int, where: str):
    """After a synced step: every layer flag holds the step's round, and each flag was
    set after the step started."""
    ptr, rnd = cache.layer_signal(g)
    flags = torch.as_tensor(_DeviceWords(ptr, layers), device=cache.device).cpu().numpy()
    assert (flags.view(np.uint32) == rnd).all(), f"{where}: flags {flags.tolist()} round {rnd}"
    ns = ula.ula_debug_layer_times(cache.ctx, g, layers)
    assert (ns[:layers] >= ns[layers]).all() and ns[layers] > 0, f"{where}: signal times {ns}"
    return ns


def unpack_bits(words: np.ndarray, nbits: int) -> np.ndarray:
    return np.unpackbits(np.ascontiguousarray(words).view(np.uint8), bitorder="little")[:nbits]


def gpu_state_in_oracle_terms(st: dict, w) -> dict:
    """Convert the library's export into the oracle's export format."""
    S, H, B = w.gpu_slots, w.host_slots, w.ring_buckets
    m = st["map"]
    tier = np.where(m == ula.MAP_UNALLOCATED, TIER_UNALLOCATED,
                    np.where(m & ula.MAP_HOST, TIER_HOST, TIER_GPU)).astype(np.uint8)
    slot = np.where(tier == TIER_UNALLOCATED, 0, m & 0x7FFFFFFF).astype(np.uint32)
    bits = np.stack([unpack_bits(st["class_bits"][c], S) for c in range(B + 2)])
    assert (bits.sum(axis=0) == 1).all(), "every GPU slot is in exactly one class"
    which = bits.argmax(axis=0)
    cls = np.where(which < B, which, np.where(which == B, COLD, FREE)).astype(np.int32)
    host_free = unpack_bits(st["host_free_bits"], H).astype(np.uint8) if H else np.zeros(0, np.uint8)
    host_owner = np.full(H, 0xFFFFFFFF, dtype=np.uint32)
    hosted = np.nonzero(tier == TIER_HOST)[0]
    host_owner[slot[hosted]] = hosted
    return {"tier": tier, "slot": slot, "cls": cls, "owner": st["owner"].copy(),
            "host_free": host_free, "host_owner": host_owner, "cur": st["cur"],
            "stamp": st["stamp"].copy(), "round": st["round"]}


def check_gpu_internal(st: dict, w):
    """Library-internal invariants: exact summaries, stamps agree with classes, counters."""
    S, H, B = w.gpu_slots, w.host_slots, w.ring_buckets
    for c in range(B + 2):
        w0, w1, w2 = st["class_bits"][c], st["class_sum1"][c], st["class_sum2"][c]
        s1 = unpack_bits(w1, len(w0))
        assert np.array_equal(s1.astype(bool), w0 != 0), f"level-1 summary of class {c}"
        s2 = unpack_bits(w2, len(w1))
        assert np.array_equal(s2.astype(bool), w1 != 0), f"level-2 summary of class {c}"
    if H:
        w0, w1, w2 = st["host_free_bits"], st["host_free_sum1"], st["host_free_sum2"]
        n0 = (H + 31) // 32
        n1 = (n0 + 31) // 32
        assert np.array_equal(unpack_bits(w1, n0).astype(bool), w0[:n0] != 0)
        assert np.array_equal(unpack_bits(w2, n1).astype(bool), w1[:n1] != 0)
    # segment counts (set bits per 1,024 slots) agree with the bitmaps
    for c in range(B + 2):
        bits = unpack_bits(st["class_bits"][c], S).astype(np.int64)
        segs = np.add.reduceat(bits, np.arange(0, S, 1024)) if S else np.zeros(0)
        assert np.array_equal(st["class_seg_count"][c][:len(segs)], segs), f"segment counts {c}"
    if H:
        bits = unpack_bits(st["host_free_bits"], H).astype(np.int64)
        segs = np.add.reduceat(bits, np.arange(0, H, 1024))
        assert np.array_equal(st["host_seg_count"][:len(segs)], segs), "host segment counts"
    r = st["round"]
    stamp = st["stamp"]
    if w.exact_lru:  # one class of occupied slots, no ring
        exp = np.where(stamp == ula.STAMP_FREE, B + 1, B)
    else:
        exp = np.where(stamp == ula.STAMP_FREE, B + 1,
                       np.where((np.uint32(r) - stamp).astype(np.uint32) >= B, B, stamp % B))
    bits = np.stack([unpack_bits(st["class_bits"][c], S) for c in range(B + 2)])
    assert np.array_equal(bits.argmax(axis=0), exp), "stamps agree with class bitmaps"
    assert st["free_gpu"] == int(bits[B + 1].sum())
    if H:
        assert st["free_host"] == int(unpack_bits(st["host_free_bits"], H).sum())


def compare_states(gpu_o: dict, orc: dict, where: str, stamps=None):
    """stamps: the oracle's (timestamps, rounds) of the group, compared when given."""
    if stamps is not None:
        orc = dict(orc, stamp=stamps[0])
        assert gpu_o["round"] == stamps[1], where
    for k in ("tier", "slot", "cls", "owner", "host_free", "host_owner") + (("stamp",) if stamps is not None else ()):
        a, b = gpu_o[k], orc[k]
        if not np.array_equal(a, b):
            idx = np.nonzero(a != b)[0][:8]
            raise AssertionError(f"{where}: {k} differs at {idx.tolist()}: gpu {a[idx].tolist()} "
                                 f"oracle {b[idx].tolist()}")
    assert gpu_o["cur"] == orc["cur"], where


def expand_id_rows(ids: np.ndarray, seed: int, g: int, j: int, W: int) -> np.ndarray:
    """Oracle id-mode rows [U][8] -> the byte rows they stand for."""
    v = ids.view(np.uint32).reshape(-1, 2)
    assert ((v[:, 1] >> 16) == g).all() and ((v[:, 1] & 0xFFFF) == j).all()
    return synth.content_list(seed, g, j, v[:, 0].copy(), W)
