"""ula_dedup_noalloc against the context's own dedup.

Some callers must not allocate device memory where they dedup a selection: a
serving engine that reserved nearly all HBM for its KV pools at start-up (a
cudaMalloc would fail or fragment the pool), or a latency-critical path that
cannot take cudaMalloc's implicit device synchronisation.  For them the library
offers ula_dedup_noalloc, whose scratch is a fixed array inside the library.

This test calls it through the C ABI and checks, entry by entry, that it gives
the same unique addresses, entry rows and count as ula_step_group's dedup, on
consecutive calls (each call starts on the scratch the previous one left).  It
lives in its own file, collected last, and needs nothing from other tests.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from synth.configs import small

pytestmark = pytest.mark.gpu


def _noalloc(ula, d_sel, stream):
    n = d_sel.numel()
    uniq = torch.full((max(n, 1),), -7, dtype=torch.int32, device=d_sel.device)
    rows = torch.full((max(n, 1),), -7, dtype=torch.int32, device=d_sel.device)
    count = torch.full((1,), -7, dtype=torch.int32, device=d_sel.device)
    stream.wait_stream(torch.cuda.current_stream(d_sel.device))  # the fills and the input
    ula.ula_dedup_noalloc(d_sel.data_ptr(), n, uniq.data_ptr(), rows.data_ptr(),
                          count.data_ptr(), stream.cuda_stream)
    stream.synchronize()
    return uniq.cpu().numpy().view(np.uint32), rows.cpu().numpy(), int(count.item())


@pytest.mark.parametrize("pads", [0.0, 0.05])
def test_noalloc_dedup_matches_step_group(pads):
    from serving_step_sparse_gb300 import ula
    from tests.gpu_harness import GpuReplay
    from tests.harness import apply_events

    w = small("longdoc").replace(pad_prob=pads, steps=3)  # 3 query tokens: duplicates across them
    assert w.entries_per_step <= ula.NOALLOC_MAX_ENTRIES
    gpu = GpuReplay(w)
    stream = torch.cuda.Stream()
    calls = 0
    try:
        for _ in range(2):
            sel, ev = gpu.trace.step()
            gpu.run_groups(sel)  # the existing entry point
            for g in range(w.n_groups):
                ref = gpu.results(g, full_out=False)
                U = int(ref["req_off"][-1])
                ref_uniq = gpu.cache.export(g)["uniq"][:U]
                uniq, rows, count = _noalloc(ula, gpu.sel_d[g].reshape(-1), stream)
                calls += 1
                assert count == U
                assert np.array_equal(rows[:sel[g].size], ref["entry_row"])
                assert np.array_equal(uniq[:U], ref_uniq)
            apply_events(gpu.alloc, gpu.free, ev)
    finally:
        gpu.close()
    assert calls >= 2


def test_noalloc_dedup_limits():
    from serving_step_sparse_gb300 import ula
    dev = torch.device("cuda")
    stream = torch.cuda.Stream()
    big = torch.zeros(ula.NOALLOC_MAX_ENTRIES + 1, dtype=torch.int32, device=dev)
    out = torch.empty_like(big)
    cnt = torch.empty(1, dtype=torch.int32, device=dev)
    with pytest.raises(ula.UlaError) as ei:
        ula.ula_dedup_noalloc(big.data_ptr(), big.numel(), out.data_ptr(), out.data_ptr(),
                              cnt.data_ptr(), stream.cuda_stream)
    assert ei.value.code == ula.ERR_CAPACITY
    # the largest size, all distinct but with repeats and pads mixed in
    n = ula.NOALLOC_MAX_ENTRIES
    rng = np.random.default_rng(5)
    vals = rng.integers(0, 40000, n, dtype=np.uint32)
    vals[rng.random(n) < 0.01] = 0xFFFFFFFF
    d = torch.from_numpy(vals.view(np.int32)).to(dev)
    uniq, rows, count = _noalloc(ula, d, stream)
    keep = vals != 0xFFFFFFFF
    exp = list(dict.fromkeys(vals[keep].tolist()))
    assert count == len(exp) and uniq[:count].tolist() == exp
    pos = {a: i for i, a in enumerate(exp)}
    assert (rows[~keep] == -1).all()
    assert rows[keep].tolist() == [pos[a] for a in vals[keep].tolist()]
