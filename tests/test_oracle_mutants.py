"""Every pin set must catch a planted mistake in the oracle (no GPU).

Each mutant is a copy of ``oracle/oracle.c`` with one plausible error
planted by text substitution (a flipped order, a reversed tie rule, an
off-by-one in the prefix match, a dropped bonus token, ...).  The copy is
compiled with gcc into a temporary directory and run against all pins; the
test passes only when at least one pin rejects the mutant.  The oracle in
the repository is never modified.
"""
import os
import shutil
import subprocess

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(os.path.abspath(oracle.__file__)), "oracle.c")

MUTANTS = {
    "value_order_flipped": [
        ("if (a->value > b->value) return -1;", "if (a->value > b->value) return 1;"),
        ("if (a->value < b->value) return 1;", "if (a->value < b->value) return -1;"),
    ],
    "tie_rule_reversed": [
        ("if (a->tie < b->tie) return -1;", "if (a->tie < b->tie) return 1;"),
        ("if (a->tie > b->tie) return 1;", "if (a->tie > b->tie) return -1;"),
    ],
    "no_tie_rule": [
        ("if (a->tie < b->tie) return -1;\n    if (a->tie > b->tie) return 1;\n", ""),
    ],
    "negative_zero_below_positive_zero": [
        ("return (double)f;", "return (f == 0.0f && (bits & 0x8000u)) ? -1e-300 : (double)f;"),
    ],
    "bit_pattern_order": [
        ("return (double)f;", "return (double)bits;"),
    ],
    "value_from_wrong_row": [
        ("out_vals[r] = col[e[r].row];", "out_vals[r] = col[r];"),
    ],
    "k_off_by_one": [
        ("for (int32_t r = 0; r < k; ++r) {", "for (int32_t r = 0; r + 1 < k; ++r) {"),
    ],
    "shortlist_ties_by_local_id": [
        ("e[i].tie = id_map ? (int64_t)id_map[i] : i;", "e[i].tie = i;"),
        ("out_ids[r] = (int32_t)e[r].tie;",
         "out_ids[r] = (int32_t)(id_map ? id_map[e[r].row] : e[r].row);"),
    ],
    "shortlist_ids_not_mapped": [
        ("out_ids[r] = (int32_t)e[r].tie;", "out_ids[r] = (int32_t)e[r].row;"),
    ],
    "argmax_last_max": [
        ("if (bf16_value(col[i]) > bf16_value(col[best])) best = i;",
         "if (bf16_value(col[i]) >= bf16_value(col[best])) best = i;"),
    ],
    "argmax_by_bits": [
        ("if (bf16_value(col[i]) > bf16_value(col[best])) best = i;",
         "if (col[i] > col[best]) best = i;"),
    ],
    "prefix_compares_next_column": [
        ("while (a < gamma && drafts[a] == t[a]) ++a;",
         "while (a < gamma && drafts[a] == t[a + 1]) ++a;"),
    ],
    "counts_all_matches_not_prefix": [
        ("while (a < gamma && drafts[a] == t[a]) ++a;",
         "for (int32_t i = 0; i < gamma; ++i) a += (drafts[i] == t[i]);"),
    ],
    "bonus_token_dropped": [
        ("commit[j] = (j <= a) ? t[j] : -1;", "commit[j] = (j < a) ? t[j] : -1;"),
    ],
    "bonus_is_draft": [
        ("commit[j] = (j <= a) ? t[j] : -1;",
         "commit[j] = (j < a) ? t[j] : ((j == a && a < gamma) ? drafts[a] : (j == a ? t[j] : -1));"),
    ],
    "padding_zero": [
        ("commit[j] = (j <= a) ? t[j] : -1;", "commit[j] = (j <= a) ? t[j] : 0;"),
    ],
    "accept_capped_below_gamma": [
        ("while (a < gamma && drafts[a] == t[a]) ++a;",
         "while (a + 1 < gamma && drafts[a] == t[a]) ++a;"),
    ],
}


def _build_mutant(tmp_path, name, subs):
    src = open(SRC).read()
    for old, new in subs:
        assert old in src, f"mutant {name}: pattern not found in oracle.c: {old!r}"
        src = src.replace(old, new)
    d = tmp_path / name
    d.mkdir()
    c = d / "oracle.c"
    c.write_text(src)
    return oracle.build(str(c), str(d / "liboracle.so"))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    lib = oracle.load(_build_mutant(tmp_path, name, MUTANTS[name]))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, oracle.OracleError, IndexError, KeyError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name!r}"
