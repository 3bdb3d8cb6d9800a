"""The library's slot-table tests catch plausible mistakes in its slot table.

Each case plants one mistake in a copy of csrc/slot_table.cpp (recency not
refreshed, the wrong victim or free slot, in-flight or pinned slots evictable,
the rank unchecked, a counter or a window edge off, a keep_score term wrong, a
release or an eviction not recorded), links the copy with the library's other
objects into a separate shared library, points the binding at it and runs the
host-only decision tests of test_abi_host.py, which compare the library with
the independent simulator: at least one must fail for every mistake. Only
host-only contexts are created, so nothing here touches a GPU.
"""
import os
import subprocess

import pytest

from rank_adapter_apply_gb300 import binding as B
from rank_adapter_apply_gb300 import build as build_mod
from tests import test_abi_host as abi

SRC = os.path.join(build_mod.CSRC, "slot_table.cpp")

# (name, text in slot_table.cpp, replacement)
MUTANTS = [
    ("touch does not refresh recency", "last_use_[slot] = ++clock_;", "++clock_;"),
    ("most recent evicted", "if (best < 0 || last_use_[s] < last_use_[best]) best = s;",
     "if (best < 0 || last_use_[s] > last_use_[best]) best = s;"),
    ("highest free slot first", "if (!occ_[i] && refs_[i] == 0) { s = i; break; }",
     "if (!occ_[i] && refs_[i] == 0) { s = i; }"),
    ("aborted slot reused while referenced", "if (!occ_[i] && refs_[i] == 0) { s = i; break; }",
     "if (!occ_[i]) { s = i; break; }"),
    ("abort allowed after the upload", "|| !occ_[slot] || !pending_[slot]) return false;",
     "|| !occ_[slot]) return false;"),
    ("in-flight slots evictable", "if (!occ_[s] || refs_[s] > 0 || pin_[s]) return false;",
     "if (!occ_[s] || pin_[s]) return false;"),
    ("pinned slots evictable", "if (!occ_[s] || refs_[s] > 0 || pin_[s]) return false;",
     "if (!occ_[s] || refs_[s] > 0) return false;"),
    ("rank not validated", "if (rank < 1 || rank > R_) {", "if (rank < 1) {"),
    ("hits not counted", "    ++hits;\n", "\n"),
    ("misses not counted", "    ++misses;\n", "\n"),
    ("thrash window one short", "epoch_ - r.last_evict_epoch <= window_) ++reloads;",
     "epoch_ - r.last_evict_epoch < window_) ++reloads;"),
    ("cooling window one short", "if (epoch_ - r.last_access_epoch < min_res_) return false;",
     "if (epoch_ - r.last_access_epoch < min_res_ - 1) return false;"),
    ("frequency window one short", "if (a.first > epoch_ - window_) n += a.second;",
     "if (a.first > epoch_ - window_ + 1) n += a.second;"),
    ("keep_score recency inverted", "const double recent = 1.0 / (1.0 + (double)(epoch_ - r.last_access_epoch));",
     "const double recent = (double)(epoch_ - r.last_access_epoch);"),
    ("keep_score frequency subtracted", "k += w_[1] * freq;", "k -= w_[1] * freq;"),
    ("keep_score priority dropped", "k += w_[2] * r.priority;", "k += 0.0;"),
    ("keep_score size added", "k -= w_[4] * rel;", "k += w_[4] * rel;"),
    ("keep_score tie to most recent", "(k == best_k && last_use_[s] < last_use_[best])",
     "(k == best_k && last_use_[s] > last_use_[best])"),
    ("release keeps the reference", "    --refs_[slot];\n", "\n"),
    ("eviction keeps the id resident", "    where_.erase(id);\n    ++evictions;", "    ++evictions;"),
    ("aborted load drops the references", "    pending_[slot] = 0;\n    where_.erase(id);\n    res_[slot] = nullptr;",
     "    pending_[slot] = 0;\n    refs_[slot] = 0;\n    where_.erase(id);\n    res_[slot] = nullptr;"),
    ("aborted load not counted", "    ++aborted_loads;\n", "\n"),
]

# host-only decision tests (library against the simulator), cheapest first
CHECKS = [
    lambda lib: abi.test_scripted_decisions_match_simulator(lib),
    lambda lib: abi.test_window_edges_and_priority_match_simulator(lib),
    lambda lib: abi.test_thrash_burst_through_abi(lib),
    lambda lib: abi.test_pinned_burst_through_abi(lib),
    lambda lib: abi.test_random_decision_log_matches_simulator(lib),
    lambda lib: abi.test_policy_decision_log_matches_simulator(lib, 0, 2),
    lambda lib: abi.test_policy_decision_log_matches_simulator(lib, 1, 0),
    lambda lib: abi.test_policy_decision_log_matches_simulator(lib, 1, 2),
    lambda lib: abi.test_assign_tokens_matches_simulator_and_maps_tokens(lib),
    lambda lib: abi.test_failed_load_leaves_the_table_consistent(lib),
    lambda lib: abi.test_late_release_after_abort_matches_simulator(lib),
    lambda lib: abi.test_serve_step_groups_and_decisions_match_simulator(lib),
    lambda lib: abi.test_random_decisions_with_aborted_loads_match_simulator(lib),
]


@pytest.fixture(scope="module")
def objects():
    """The real library's object files (built once), slot_table.cpp's left out."""
    build_mod.build()
    objs = [os.path.join(build_mod.BUILD, s + ".o") for s in build_mod.SOURCES if s != "slot_table.cpp"]
    assert all(os.path.exists(o) for o in objs)
    return objs


def _link(text, objs, out_dir):
    src = os.path.join(out_dir, "slot_table.cpp")
    with open(src, "w") as f:
        f.write(text)
    nvcc = build_mod._nvcc()
    obj = os.path.join(out_dir, "slot_table.o")
    lib = os.path.join(out_dir, "librank_adapter_apply_mutant.so")
    subprocess.run([nvcc, *build_mod.FLAGS, f"-I{build_mod.CSRC}", "-x", "c++", "-c", src, "-o", obj],
                   check=True, capture_output=True)
    subprocess.run([nvcc, *build_mod.ARCH, "-shared", "-cudart", "static", *objs, obj, "-o", lib],
                   check=True, capture_output=True)
    return lib


def _first_failing_check(monkeypatch, lib_path):
    monkeypatch.setattr(B, "_lib", None)
    lib = B.load(lib_path)
    for i, check in enumerate(CHECKS):
        try:
            check(lib)
        except (AssertionError, B.LoraError):
            return i
    return None


def test_unchanged_copy_passes_every_check(objects, tmp_path, monkeypatch):
    lib = _link(open(SRC).read(), objects, str(tmp_path))
    assert _first_failing_check(monkeypatch, lib) is None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_check(name, old, new, objects, tmp_path, monkeypatch):
    text = open(SRC).read()
    assert text.count(old) == 1, f"{old!r} is not unique in slot_table.cpp"
    lib = _link(text.replace(old, new), objects, str(tmp_path))
    assert _first_failing_check(monkeypatch, lib) is not None, f"no check catches: {name}"
