"""The oracle's pins catch plausible mistakes in the oracle itself.

Each case below plants one mistake in a copy of the C oracle (a dropped term, a
wrong sign, index or slot, a transposed operand, an off-by-one loop bound, a
rounded intermediate, a wrong scale), builds the copy with the oracle's own
compiler flags, points the oracle module at it and runs the pins of
test_oracle_pins.py: at least one pin must fail for every mistake. Every
planted index stays inside the arrays it reads, so no copy can crash.
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
