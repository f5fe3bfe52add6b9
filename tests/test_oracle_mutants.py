"""Plant plausible mistakes in a private copy of the C oracle and check that the
pins catch every one of them.

Each mutant is the oracle source with one textual edit (a dropped term, a wrong
index, a wrong reading of shard ownership), compiled to a temporary library on
the CPU.  The pins of ``test_oracle_pins`` are run against it; at least one
must fail.  The committed oracle is never modified.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_causal_pins as cpins
import test_oracle_pins as pins
import test_oracle_varlen_pins as vpins

MUTANTS = {
    "scale dropped": ("x[j] = scale * dot;", "x[j] = dot;"),
    "no normalisation": ("orow[d] /= l;", "orow[d] /= 1.0;"),
    "sum of weights wrong": ("l += x[j];", "l += x[j] * x[j];"),
    "value row from the query index": ("const double* vj = vd + j * D;",
                                       "const double* vj = vd + (j == 0 ? 0 : j - 1) * D;"),
    "strided sequence ownership": ("idx4(b, p * Sl + s2, j, d, S, Hl, D)];\n    return 0;\n}\n\n/*\n * The inverse",
                                   "idx4(b, s2 * P + p, j, d, S, Hl, D)];\n    return 0;\n}\n\n/*\n * The inverse"),
    "local head index in the destination": (
        "out[(size_t)(p * B * Sl * H * D) + idx4(b, s2, r * Hl + j, d, Sl, H, D)] =\n"
        "                                L[",
        "out[(size_t)(p * B * Sl * H * D) + idx4(b, s2, j * P + r, d, Sl, H, D)] =\n"
        "                                L["),
    "head shard takes the wrong head": ("o[idx4(b, s, r * Hl + j, d, S, H, D)];",
                                        "o[idx4(b, s, j * P + r, d, S, H, D)];"),
}

# Mistakes in the causal key window (row i must see keys 0 .. i), caught by the
# causal pins of test_oracle_causal_pins.
CAUSAL_SITE = "return causal ? i + 1 : S;"
CAUSAL_MUTANTS = {
    "causal window one key short": "return causal ? (i > 0 ? i : 1) : S;",
    "causal window one key long": "return causal ? (i + 2 < S ? i + 2 : S) : S;",
    "causal window counted from the end": "return causal ? S - i : S;",
    "causal flag ignored": "return S;",
}

CAUSAL_PIN_CASES = [
    (cpins.test_causal_worked_example_by_hand, ()),
    (cpins.test_causal_first_row_copies_first_value_row, (5,)),
    (cpins.test_causal_q_zero_gives_prefix_means_of_v, (7,)),
    (cpins.test_causal_last_row_equals_bidirectional, ()),
    (cpins.test_causal_future_keys_and_values_do_not_matter, ()),
    (cpins.test_causal_weights_vanish_above_the_diagonal_and_sum_to_one, ()),
    (cpins.test_causal_brute_force_numpy, (8,)),
    (cpins.test_causal_torch_sdpa_fp64_crosscheck, ()),
]

PIN_CASES = [
    (pins.test_worked_example_by_hand, ()),
    (pins.test_reshard_index_table_by_hand, ()),
    (pins.test_head_shards_hold_contiguous_head_ranges, ()),
    (pins.test_brute_force_numpy, (8, 2)),
    (pins.test_q_zero_gives_mean_of_v, (7,)),
    (pins.test_weights_sum_to_one_and_match_output, ()),
    (pins.test_key_permutation_invariance, ()),
    (pins.test_reshard_of_one_hot_layout_inputs, ()),
    (pins.test_torch_sdpa_fp64_crosscheck, ()),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation site for {name!r} not unique"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(lib),
                    str(path), "-lm"], check=True)
    return str(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path, monkeypatch):
    lib_path = _build_mutant(tmp_path, name, *MUTANTS[name])
    monkeypatch.setattr(oracle, "_LIB", lib_path)
    monkeypatch.setattr(oracle, "_SRC", lib_path)  # keep build() from rebuilding
    monkeypatch.setattr(oracle, "_lib", None)
    failures = []
    for fn, args in PIN_CASES:
        try:
            fn(*args)
        except AssertionError:
            failures.append(fn.__name__)
    monkeypatch.setattr(oracle, "_lib", None)
    assert failures, f"no pin caught the mutant {name!r}"


@pytest.mark.parametrize("name", sorted(CAUSAL_MUTANTS))
def test_causal_pins_catch_mutant(name, tmp_path, monkeypatch):
    lib_path = _build_mutant(tmp_path, name, CAUSAL_SITE, CAUSAL_MUTANTS[name])
    monkeypatch.setattr(oracle, "_LIB", lib_path)
    monkeypatch.setattr(oracle, "_SRC", lib_path)
    monkeypatch.setattr(oracle, "_lib", None)
    failures = []
    for fn, args in CAUSAL_PIN_CASES:
        try:
            fn(*args)
        except (AssertionError, RuntimeError):
            failures.append(fn.__name__)
    monkeypatch.setattr(oracle, "_lib", None)
    assert failures, f"no causal pin caught the mutant {name!r}"


# Mistakes in the packed variable-length form (a Python function over the C
# row routine), planted by wrapping the committed function.
_varlen = oracle.attention_varlen


def _boundary_shifted(q, k, v, seqlens, scale, causal=False, nthreads=None):
    lens = list(seqlens)
    i = next((j for j in range(len(lens) - 1) if lens[j] > 1), None)
    if i is not None:   # first boundary one row late
        lens[i] -= 1
        lens[i + 1] += 1
    return _varlen(q, k, v, lens, scale, causal, nthreads)


VARLEN_MUTANTS = {
    "boundary one row off": _boundary_shifted,
    "rows attend across sequences": lambda q, k, v, seqlens, scale, causal=False, nthreads=None:
        _varlen(q, k, v, [sum(seqlens)], scale, causal, nthreads),
    "causal flag dropped": lambda q, k, v, seqlens, scale, causal=False, nthreads=None:
        _varlen(q, k, v, seqlens, scale, False, nthreads),
}

VARLEN_PIN_CASES = [
    (vpins.test_varlen_worked_example_by_hand, (True,)),
    (vpins.test_varlen_brute_force_numpy, ([5, 1, 7], True)),
    (vpins.test_varlen_torch_sdpa_fp64_crosscheck, (False,)),
    (vpins.test_varlen_other_and_empty_sequences_do_not_matter, ()),
    (vpins.test_varlen_q_zero_gives_sequence_means, (True,)),
]


@pytest.mark.parametrize("name", sorted(VARLEN_MUTANTS))
def test_varlen_pins_catch_mutant(name, monkeypatch):
    monkeypatch.setattr(oracle, "attention_varlen", VARLEN_MUTANTS[name])
    failures = []
    for fn, args in VARLEN_PIN_CASES:
        try:
            fn(*args)
        except AssertionError:
            failures.append(fn.__name__)
    assert failures, f"no varlen pin caught the mutant {name!r}"


def test_unmutated_copy_passes_all_pins(tmp_path, monkeypatch):
    src = open(oracle._SRC).read()
    lib_path = _build_mutant(tmp_path, "identity", "double m = -INFINITY;", "double m = -INFINITY;")
    monkeypatch.setattr(oracle, "_LIB", lib_path)
    monkeypatch.setattr(oracle, "_SRC", lib_path)
    monkeypatch.setattr(oracle, "_lib", None)
    for fn, args in PIN_CASES + CAUSAL_PIN_CASES + VARLEN_PIN_CASES:
        fn(*args)
    monkeypatch.setattr(oracle, "_lib", None)
    assert "double m = -INFINITY;" in src
    assert isinstance(ctypes.CDLL(lib_path), ctypes.CDLL)
