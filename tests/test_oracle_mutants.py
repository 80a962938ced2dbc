"""Planted mistakes in the oracle (CPU only).

Each mutant is one plausible slip in the oracle's C source: a dropped term,
a wrong sign, index or constant, a transposed operand, a flipped comparison,
a skipped step.  The test makes it in a text copy of the source, compiles the
copy with the oracle's own flags into a temporary library, and swaps that
library in for the oracle's.  The pins in test_oracle_pins.py must then
reject it: each mutant names the pins expected to catch it, and at least one
of them has to fail.  Every mutant keeps its memory accesses in bounds, so a
survivor shows up as a failed test, never as a crash.
"""

import ctypes
import os

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "snack_oracle.c")

# the pins, by name, with the arguments a parametrised one is called with
PIN = {
    "brute": lambda: (pins.test_dense_brute_force_tiny(7, 33, 3), pins.test_dense_brute_force_tiny(33, 7, 8)),
    "3x3": pins.test_every_3x3_pattern,
    "dense": pins.test_zero_sparsity_is_dense_gemm,
    "identity": pins.test_identity_weight,
    "fd": pins.test_finite_differences,
    "adjoint": pins.test_linearity_and_adjointness,
    "coo": pins.test_out_of_range_rejected,
    "gelu": pins.test_gelu_pins,
    "kat": pins.test_splitmix64_known_answers,
    "stream": pins.test_draw_stream_is_splitmix64_from_state_zero,
    "rs_inv": pins.test_restructure_invariants_random,
    "rs_3x3": pins.test_restructure_every_3x3_pattern,
    "rs_ties": pins.test_restructure_ties_and_nan_order,
    "rs_uniform": pins.test_regrow_uniform_over_empty_positions,
    "rows_one": pins.test_rows_one_row_equals_unstructured,
    "rows_base": pins.test_rows_stream_base,
    "rows_inv": pins.test_rows_invariants_random,
    "rows_3x3": pins.test_rows_every_3x3_pattern,
}

# (name, text in the source, replacement, pins expected to catch it)
MUTANTS = [
    ("fwd drops the bias", "yb[r] = c->bias ? c->bias[r] : 0.0;", "yb[r] = 0.0;", ["brute", "fd"]),
    ("fwd gathers the mirrored X column", "double term = c->val[k] * xb[c->col[k]];",
     "double term = c->val[k] * xb[c->in_f - 1 - c->col[k]];", ["brute", "3x3", "identity"]),
    ("fwd subtracts the terms", "yb[c->row[k]] += term;", "yb[c->row[k]] -= term;", ["brute", "identity"]),
    ("fwd sums signed terms into T", "if (tb) tb[c->row[k]] += fabs(term);", "if (tb) tb[c->row[k]] += term;",
     ["brute", "3x3"]),
    ("dx gathers the mirrored dY row", "double term = c->val[k] * g[c->row[k]];",
     "double term = c->val[k] * g[c->out_f - 1 - c->row[k]];", ["brute", "3x3", "adjoint"]),
    ("dx scatters to the mirrored column", "o[c->col[k]] += term;", "o[c->in_f - 1 - c->col[k]] += term;",
     ["brute", "identity", "fd"]),
    ("dw pairs dY with the mirrored X column", "c->x[b * c->in_f + c->col[k]]",
     "c->x[b * c->in_f + (c->in_f - 1 - c->col[k])]", ["brute", "fd", "adjoint"]),
    ("dw skips the last batch row", "for (int64_t b = 0; b < c->batch; ++b) {",
     "for (int64_t b = 0; b + 1 < c->batch; ++b) {", ["brute", "fd"]),
    ("db skips the last batch row", "for (int64_t b = 0; b < c->batch; ++b) s += c->dy[b * c->out_f + r];",
     "for (int64_t b = 0; b + 1 < c->batch; ++b) s += c->dy[b * c->out_f + r];", ["brute", "fd"]),
    ("coo check accepts repeated positions", "if (!(a < b)) return 2;", "if (!(a <= b)) return 2;", ["coo"]),
    ("GELU with erf(x / 2)", "return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }",
     "return 0.5 * x * (1.0 + erf(x / 2.0)); }", ["gelu"]),
    ("GELU' drops x phi(x)", " + x * inv_sqrt_2pi * exp(-0.5 * x * x);", ";", ["gelu"]),
    ("GELU' with exp(-x^2)", "exp(-0.5 * x * x)", "exp(-x * x)", ["gelu"]),
    ("mix shifts by 31 first", "z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;",
     "z = (z ^ (z >> 31)) * 0xBF58476D1CE4E5B9ULL;", ["kat", "stream"]),
    ("stream increment off by two", "static const uint64_t SM64_GAMMA = 0x9E3779B97F4A7C15ULL;",
     "static const uint64_t SM64_GAMMA = 0x9E3779B97F4A7C13ULL;", ["stream"]),
    ("draw i from state + i * gamma", "oracle_regrow_base(seed, step) + (i + 1) * SM64_GAMMA",
     "oracle_regrow_base(seed, step) + i * SM64_GAMMA", ["stream"]),
    ("base mixes step with the mixed seed", "return oracle_splitmix64_mix(seed ^ oracle_splitmix64_mix(step));",
     "return oracle_splitmix64_mix(step ^ oracle_splitmix64_mix(seed));", ["rows_one", "rows_base"]),
    ("prune the largest magnitudes", "return a->mag < b->mag ? -1 : 1;", "return a->mag > b->mag ? -1 : 1;",
     ["rs_inv", "rs_3x3", "rs_ties"]),
    ("ties pruned from the back", "return a->k < b->k ? -1 : (a->k > b->k ? 1 : 0);",
     "return a->k > b->k ? -1 : (a->k < b->k ? 1 : 0);", ["rs_inv", "rs_3x3", "rs_ties"]),
    ("NaN pruned before numbers", "return a->is_nan < b->is_nan ? -1 : 1;",
     "return a->is_nan > b->is_nan ? -1 : 1;", ["rs_inv", "rs_ties"]),
    ("signed value instead of magnitude", "keys[k].mag = keys[k].is_nan ? 0.0 : fabs(val[k]);",
     "keys[k].mag = keys[k].is_nan ? 0.0 : val[k];", ["rs_inv", "rs_3x3", "rs_ties"]),
    ("regrow at stored positions", "    if (sorted_contains(pos, nnz, p)) continue;\n", "",
     ["rs_inv", "rs_3x3", "rs_uniform"]),
    ("regrow one position twice", "if (!pos_set_insert(&acc, p)) continue;", "pos_set_insert(&acc, p);",
     ["rs_inv", "rs_3x3"]),
    ("regrown position split by out_f", "row_out[j] = (int32_t)(grown[g] / (uint64_t)in_f);\n"
     "        col_out[j] = (int32_t)(grown[g] % (uint64_t)in_f);",
     "row_out[j] = (int32_t)(grown[g] % (uint64_t)out_f);\n"
     "        col_out[j] = (int32_t)(grown[g] / (uint64_t)out_f);", ["rs_inv"]),
    ("merge puts regrown first", "if (have_a && (!have_g || pos[a] < grown[g])) {",
     "if (have_a && (!have_g || pos[a] > grown[g])) {", ["rs_inv", "rs_3x3"]),
    ("regrown positions left unsorted", "  qsort(grown, (size_t)n_prune, sizeof(uint64_t), cmp_u64);\n", "",
     ["rs_inv", "rs_3x3"]),
    ("row stream constant off by two", "static const uint64_t ROW_STREAM_K = 0xD1B54A32D192ED03ULL;",
     "static const uint64_t ROW_STREAM_K = 0xD1B54A32D192ED05ULL;", ["rows_base"]),
    ("row stream ignores the row", "oracle_splitmix64_mix(step ^ (r * ROW_STREAM_K))",
     "oracle_splitmix64_mix(step)", ["rows_base"]),
    ("row draws scaled to in_f - 1", "(unsigned __int128)(uint64_t)in_f) >> 64",
     "(unsigned __int128)(uint64_t)(in_f - 1)) >> 64", ["rows_one"]),
    ("row regrows a column twice", "      if (dup) continue;\n", "", ["rows_inv", "rows_3x3"]),
    ("row regrows stored columns", "      if (sorted_contains(rowpos, len, c)) continue;\n", "",
     ["rows_inv", "rows_3x3", "rows_one"]),
    ("row merge puts regrown first", "(uint64_t)col[a] < grown[g]", "(uint64_t)col[a] > grown[g]",
     ["rows_inv", "rows_3x3", "rows_one"]),
]


def test_mutant_list_matches_the_source():
    src = open(SRC).read()
    for name, old, _, pin_names in MUTANTS:
        assert src.count(old) == 1, name  # each slip is made at exactly one place
        assert pin_names and all(p in PIN for p in pin_names), name
    assert len({m[0] for m in MUTANTS}) == len(MUTANTS)


@pytest.mark.parametrize("name,old,new,pin_names", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, monkeypatch, name, old, new, pin_names):
    src = open(SRC).read()
    assert src.count(old) == 1
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib_path = str(tmp_path / "libmutant.so")
    oracle.compile_library(str(path), lib_path)
    monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(lib_path)))
    caught = []
    for p in pin_names:
        try:
            PIN[p]()
        except (Exception, pytest.fail.Exception) as e:  # a failed assertion or pytest.raises, an oracle error
            caught.append(f"{p}: {type(e).__name__}")
    assert caught, f"mutant '{name}' passed the pins {pin_names}"


def test_unmodified_copy_passes_every_pin(tmp_path, monkeypatch):
    # control: the same copy-compile-swap path without a slip passes all the
    # pins above, so the mutants fail for their slip alone
    path = tmp_path / "copy.c"
    path.write_text(open(SRC).read())
    lib_path = str(tmp_path / "libcopy.so")
    oracle.compile_library(str(path), lib_path)
    monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(lib_path)))
    for p in PIN.values():
        p()
