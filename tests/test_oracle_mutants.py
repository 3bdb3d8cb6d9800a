"""The oracle's pins catch plausible mistakes in the oracle itself.

Each case below plants one mistake in a copy of the C oracle (a dropped term, a
wrong sign, index or slot, a transposed operand, an off-by-one loop bound, a
rounded intermediate, a wrong scale), builds the copy with the oracle's own
compiler flags, points the oracle module at it and runs the pins of
test_oracle_pins.py: at least one pin must fail for every mistake. Every
planted index stays inside the arrays it reads, so no copy can crash. The
second half does the same for the slot-table simulator (recency, victim
choice, in-flight and pinned slots, rank check, counters, window edges and
every keep_score term) against the hand-derived scripts of test_lru_sim.py.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "lora_oracle.c")

# (name, text in the oracle, replacement, which occurrence (0 = first))
MUTANTS = [
    ("y_in term dropped", "out[i] = elem(y_in, dtype, (size_t)t * d_out + i);", "out[i] = 0.0;", 0),
    ("delta subtracted", "out[i] += scale * acc;", "out[i] -= scale * acc;", 0),
    ("scale dropped", "double scale = alpha[s] / (double)r;", "double scale = 1.0;", 0),
    ("scale over max_lora_rank", "double scale = alpha[s] / (double)r;", "double scale = alpha[s] / (double)R;", 0),
    ("scale times rank", "double scale = alpha[s] / (double)r;", "double scale = alpha[s] * (double)r;", 0),
    ("alpha of slot 0", "double scale = alpha[s] / (double)r;", "double scale = alpha[0] / (double)r;", 0),
    ("rank of slot 0", "int r = rank[s];", "int r = rank[0] > 0 ? rank[0] : 1;", 0),
    ("A of slot 0", "size_t arow = ((size_t)s * R + k) * (size_t)d_in;",
     "size_t arow = ((size_t)0 * R + k) * (size_t)d_in;", 0),
    ("B of slot 0", "size_t brow = ((size_t)s * d_out + i) * (size_t)R;",
     "size_t brow = ((size_t)0 * d_out + i) * (size_t)R;", 0),
    ("A transposed within its slot", "acc += elem(A_pool, dtype, arow + j)",
     "acc += elem(A_pool, dtype, (size_t)s * R * d_in + ((size_t)j * R + k) % ((size_t)R * d_in))", 0),
    ("B transposed within its slot", "acc += elem(B_pool, dtype, brow + k)",
     "acc += elem(B_pool, dtype, (size_t)s * d_out * R + ((size_t)k * d_out + i) % ((size_t)R * d_out))", 0),
    ("x row of the list position", "elem(x, dtype, (size_t)t * d_in + j)", "elem(x, dtype, (size_t)n * d_in + j)", 0),
    ("y_in row of the list position", "elem(y_in, dtype, (size_t)t * d_out + i)",
     "elem(y_in, dtype, (size_t)n * d_out + i)", 0),
    ("output column reversed", "out[i] += scale * acc;", "out[d_out - 1 - i] += scale * acc;", 0),
    ("last rank dropped in the shrink", "for (int k = 0; k < kmax; k++)", "for (int k = 0; k < kmax - 1; k++)", 0),
    ("last rank dropped in the expand", "for (int k = 0; k < kmax; k++)", "for (int k = 0; k < kmax - 1; k++)", 1),
    ("last input column dropped", "for (int j = 0; j < d_in; j++)", "for (int j = 0; j < d_in - 1; j++)", 0),
    ("intermediate rounded to fp32", "v[k] = acc;", "v[k] = (float)acc;", 0),
    ("bf16 decoded with a wrong shift", "<< 16;", "<< 15;", 0),
    ("empty slots applied", "if (s < 0 || s >= S || rank[s] <= 0)", "if (s < 0 || s >= S)", 0),
    ("base-only token applied as slot 0", "int s = token_slot_idx[t];",
     "int s = token_slot_idx[t] < 0 ? 0 : token_slot_idx[t];", 0),
]

# cheap pins first; the first failure ends a case
PINS = [pins.test_golden_peft_example, pins.test_merged_weight_identity_exact,
        pins.test_rank_one_one_hot, pins.test_invalid_and_empty_slots_are_noops,
        pins.test_scale_uses_true_rank_and_is_linear_in_alpha,
        pins.test_library_reduction_single_slot, pins.test_merged_weight_identity_random_bf16,
        pins.test_zero_B_and_minus_one_reproduce_base, pins.test_bf16_decoding_is_exact,
        pins.test_token_list_matches_whole_batch, pins.test_zero_padding_is_bit_exact]


def _replace_nth(text, old, new, n):
    at = -1
    for _ in range(n + 1):
        at = text.find(old, at + 1)
        assert at >= 0, f"{old!r}: fewer than {n + 1} occurrences in the oracle"
    return text[:at] + new + text[at + len(old):]


def _build(src_text, out_dir):
    src = os.path.join(out_dir, "mutant.c")
    lib = os.path.join(out_dir, "libmutant.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    "-fno-fast-math", "-std=c11", src, "-o", lib], check=True)
    return lib


def _first_failing_pin():
    for pin in PINS:
        try:
            pin()
        except (AssertionError, RuntimeError):
            return pin.__name__
    return None


@pytest.fixture
def use_library(monkeypatch):
    """Point the oracle module at another build of its C source."""
    def use(path):
        monkeypatch.setattr(oracle, "_lib", None)
        monkeypatch.setattr(oracle, "build", lambda force=False: path)
    yield use
    oracle._lib = None


def test_unchanged_copy_passes_every_pin(tmp_path, use_library):
    use_library(_build(open(SRC).read(), str(tmp_path)))
    assert _first_failing_pin() is None


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, old, new, nth, tmp_path, use_library):
    text = open(SRC).read()
    mutant = _replace_nth(text, old, new, nth)
    assert mutant != text
    use_library(_build(mutant, str(tmp_path)))
    assert _first_failing_pin() is not None, f"no pin catches: {name}"


# ---- the slot-table simulator ------------------------------------------------

import importlib.util  # noqa: E402
import sys  # noqa: E402

from tests import test_lru_sim as lru_pins  # noqa: E402

SIM_SRC = os.path.join(os.path.dirname(oracle.__file__), "lru_sim.py")

SIM_MUTANTS = [
    ("touch does not refresh recency", "self.last_use[s] = self.clock", "self.last_use[s] = self.last_use[s]", 0),
    ("most recent evicted", "return min(cands, key=lambda s: self.last_use[s])",
     "return max(cands, key=lambda s: self.last_use[s])", 0),
    ("highest free slot first", "s = free[0]", "s = free[-1]", 0),
    ("in-flight adapters evictable", "if aid is None or self.refs[s] > 0 or self.pinned[s]:",
     "if aid is None or self.pinned[s]:", 0),
    ("pinned adapters evictable", "if aid is None or self.refs[s] > 0 or self.pinned[s]:",
     "if aid is None or self.refs[s] > 0:", 0),
    ("rank not validated", "if rank < 1 or rank > self.R:", "if rank < 1:", 0),
    ("hits not counted", "self.hits += 1", "self.hits += 0", 0),
    ("hit does not touch", "self._touch(s)", "pass", 0),
    ("reloads never counted", "self.reloads += 1", "self.reloads += 0", 0),
    ("thrash window one short", "self.epoch - rec.last_evict_epoch <= self.window",
     "self.epoch - rec.last_evict_epoch < self.window", 0),
    ("thrash window unbounded", "self.epoch - rec.last_evict_epoch <= self.window", "True", 0),
    ("cooling window ignored", "if self.min_residency > 0 and", "if False and", 0),
    ("cooling window one short", "< self.min_residency:", "< self.min_residency - 1:", 0),
    ("release keeps the reference", "self.refs[s] -= 1", "self.refs[s] -= 0", 0),
    ("keep_score frequency subtracted", "k += w2 * freq", "k -= w2 * freq", 0),
    ("keep_score recency inverted", "recent = 1.0 / (1.0 + float(self.epoch - rec.last_access))",
     "recent = float(self.epoch - rec.last_access)", 0),
    ("keep_score priority dropped", "k += w3 * rec.priority", "k += 0.0", 0),
    ("keep_score size added", "k -= w5 * rel", "k += w5 * rel", 0),
    ("keep_score highest evicted", "return min(cands, key=lambda s: (self.keep_score(s), self.last_use[s]))",
     "return max(cands, key=lambda s: (self.keep_score(s), self.last_use[s]))", 0),
    ("keep_score tie to most recent", "return min(cands, key=lambda s: (self.keep_score(s), self.last_use[s]))",
     "return min(cands, key=lambda s: (self.keep_score(s), -self.last_use[s]))", 0),
    ("frequency window one short", "if e > self.epoch - self.window)", "if e > self.epoch - self.window + 1)", 0),
    ("pin of an empty slot accepted", "if self.slot_id[s] is None:\n            return STATE_ERR",
     "if False:\n            return STATE_ERR", 0),
    ("aborted load keeps the id resident", "del self.where[aid]\n        self.aborted += 1",
     "self.aborted += 1", 0),
    ("aborted load drops the references", "del self.where[aid]\n        self.aborted += 1",
     "self.refs[s] = 0\n        del self.where[aid]\n        self.aborted += 1", 0),
    ("abort allowed after the upload", "if aid is None or not self.pending[s]:", "if aid is None:", 0),
    ("aborted slot reused while referenced", "if self.slot_id[s] is None and self.refs[s] == 0]",
     "if self.slot_id[s] is None]", 0),
    ("upload does not clear pending", "self.pending[s] = False\n        return OK", "return OK", 0),
]

LRU_PINS = [getattr(lru_pins, n) for n in dir(lru_pins) if n.startswith("test_")]


def _load_sim(text, out_dir, tag):
    path = os.path.join(out_dir, f"lru_sim_{tag}.py")
    with open(path, "w") as f:
        f.write(text)
    name = f"lru_sim_{tag}"
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod              # dataclasses look their module up while the class is built
    try:
        spec.loader.exec_module(mod)
    finally:
        del sys.modules[name]
    return mod


def _first_failing_lru_pin(monkeypatch, mod):
    monkeypatch.setattr(lru_pins, "LruSlotSim", mod.LruSlotSim)
    for pin in LRU_PINS:
        try:
            pin()
        except (AssertionError, KeyError, IndexError, TypeError, ValueError):
            return pin.__name__
    return None


def test_unchanged_simulator_passes_every_pin(tmp_path, monkeypatch):
    assert len(LRU_PINS) >= 14
    mod = _load_sim(open(SIM_SRC).read(), str(tmp_path), "same")
    assert _first_failing_lru_pin(monkeypatch, mod) is None


@pytest.mark.parametrize("name,old,new,nth", SIM_MUTANTS, ids=[m[0] for m in SIM_MUTANTS])
def test_planted_simulator_mistake_fails_a_pin(name, old, new, nth, tmp_path, monkeypatch):
    text = open(SIM_SRC).read()
    mutant = _replace_nth(text, old, new, nth)
    assert mutant != text
    mod = _load_sim(mutant, str(tmp_path), "mut")
    assert _first_failing_lru_pin(monkeypatch, mod) is not None, f"no pin catches: {name}"
