"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle source (on the CPU), builds
it, runs a fast subset of the pins against it and expects at least one to fail.
"""
from __future__ import annotations

import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_oracle_tp as tp_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ula_oracle.cpp")

# (name, original text, planted mistake)
MUTATIONS = [
    ("ring newest first", "take(g.ring[(g.cur + d) % o->B], (int)((g.cur + d) % o->B));",
     "take(g.ring[(g.cur + o->B - d) % o->B], (int)((g.cur + o->B - d) % o->B));"),
    ("no fold into cold", "for (uint32_t s : g.ring[g.cur]) {", "for (uint32_t s : std::set<uint32_t>{}) {"),
    ("cold after ring", "    take(g.cold, kCold);\n    for (uint32_t d = 1; d < o->B; ++d) take(g.ring[(g.cur + d) % o->B], (int)((g.cur + d) % o->B));",
     "    for (uint32_t d = 1; d < o->B; ++d) take(g.ring[(g.cur + d) % o->B], (int)((g.cur + d) % o->B));\n    take(g.cold, kCold);"),
    ("highest slot first", "    for (uint32_t s : from) {\n      if (victims.size() == M) return;",
     "    for (auto it = from.rbegin(); it != from.rend(); ++it) { uint32_t s = *it;\n      if (victims.size() == M) return;"),
    ("write-back to highest free host slot", "  for (uint32_t hs : g.host_free) {\n    if (wb_host.size()",
     "  for (auto it = g.host_free.rbegin(); it != g.host_free.rend(); ++it) { uint32_t hs = *it;\n    if (wb_host.size()"),
    ("evicted owner's map not updated", "      g.where[prev_owner] = Location{kOnHost, hs};\n", ""),
    ("misses paired in reverse", "    const uint32_t a = misses[i];", "    const uint32_t a = misses[M - 1 - i];"),
    ("rotation skips a bucket", "  g.cur = (g.cur + 1) % o->B;", "  g.cur = (g.cur + 2) % o->B;"),
    ("gather always reads layer 0", "&pool[(size_t)loc.slot * sb + (size_t)j * o->row_bytes]",
     "&pool[(size_t)loc.slot * sb + (size_t)0 * o->row_bytes]"),
    ("bypass keeps the last misses instead of the first", "    misses.resize(can_place);",
     "    misses.erase(misses.begin(), misses.end() - can_place);"),
    ("miss host slots never released", "  for (uint32_t hs : released_host) {\n    g.host_free.insert(hs);", "  for (uint32_t hs : released_host) {\n"),
    ("alloc takes highest free slot", "      if (!g.free_slots.empty()) {  // lowest free GPU slot; a prefill write counts as an access\n        uint32_t s = *g.free_slots.begin();",
     "      if (!g.free_slots.empty()) {\n        uint32_t s = *g.free_slots.rbegin();"),
    ("hits not marked as accessed", "    if (g.where[a].tier == kOnGpu) touch(*o, g, g.where[a].slot);", "    (void)a;"),
    ("write-back skipped (data lost)", "      std::memcpy(&g.host_pool[(size_t)hs * sb], &g.gpu_pool[(size_t)v * sb], sb);\n", ""),
    ("fill skipped", "    std::memcpy(&g.gpu_pool[(size_t)v * sb], &g.host_pool[(size_t)src_host * sb], sb);\n    g.where[a]",
     "    g.where[a]"),
    ("exact LRU: occupied slots taken in slot order, not oldest first",
     "    for (const auto &ts : g.by_age) {\n      if (victims.size() == M || ts.first == g.round) break;\n      victims.push_back(ts.second);",
     "    for (uint32_t sl : g.cold) {\n      if (victims.size() == M) break;\n      if (g.stamp[sl] == g.round) continue;\n      victims.push_back(sl);"),
    ("exact LRU: an access renews the timestamp but not the age order",
     "    g.by_age.insert({g.round, s});\n  } else {",
     "    g.by_age.insert({g.stamp[s] == kNone ? g.round : g.stamp[s], s});\n  } else {"),
    ("timestamps of alloc placements one round late", "  g.stamp[s] = g.round;\n}",
     "  g.stamp[s] = g.round + (g.owner[s] == kNone ? 1u : 0u);\n}"),
    ("TP buffer: ring newest first", "take(b.ring[(b.cur + d) % t->B], (int)((b.cur + d) % t->B));",
     "take(b.ring[(b.cur + t->B - d) % t->B], (int)((b.cur + t->B - d) % t->B));"),
    ("TP buffer: evicted copy still mapped", "      if (b.owner[v] != kNone) b.where[b.owner[v]] = -1;  // the copy is dropped\n", ""),
    ("TP fetch from the neighbouring partition", "      const Oracle *o = t->parts[a % P];",
     "      const Oracle *o = t->parts[(a + 1) % P];"),
]


def _fast_pins():
    pins.test_worked_example_golden()
    for seed in range(0, 80, 9):
        pins.test_overflow_bypass_matches_timestamp_model(seed)
    for seed in range(0, 120, 7):
        pins.test_with_folds_matches_timestamp_model(seed)
    for seed in range(0, 60, 9):
        pins.test_no_fold_equals_round_lru(seed)
    for seed in range(0, 120, 7):
        pins.test_exact_lru_matches_timestamp_model(seed)
    for seed in range(0, 40, 5):
        pins.test_exact_lru_bypass_matches_timestamp_model(seed)
    for seed in range(0, 60, 6):
        tp_pins.test_tp_buffer_matches_timestamp_model(seed)
    tp_pins.test_tp_one_partition_is_the_dp_oracle()
    pins.test_rotation_only_relabels()
    pins.test_errors_leave_state_untouched()
    pins.test_alloc_placement_and_free()
    pins.test_workload_closed_forms_and_invariants("tiny_1x4k")
    pins.test_workload_closed_forms_and_invariants("longdoc")


def test_unmutated_source_passes():
    _fast_pins()


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new, monkeypatch, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {name}"
    mutated = tmp_path / "mut.cpp"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", "-o", str(so), str(mutated)],
                   check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.load_variant(str(so)))
    caught = False
    try:
        _fast_pins()
    except (AssertionError, oracle.OracleError):
        caught = True
    assert caught, f"planted mistake '{name}' passed every pin"
