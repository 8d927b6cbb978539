"""Mutation tests: plausible one-line mistakes planted in a temporary copy of
the oracle source must each make at least one pin fail.  This shows the pins
are not vacuous (the same check the mask kernel's authors ran with two
kernel mutants, prhub report on vLLM PR #56628, implementation notes)."""
import os

import pytest

import oracle
from tests import test_combine_window as combine
from tests import test_oracle_attention as att
from tests import test_oracle_pins as pins
from tests.common import load_golden

# (name, exact text in dsa_oracle.c, replacement)
MUTANTS = [
    ("key_keeps_negative_bits", "(u & 0x80000000u) ? ~u : (u | 0x80000000u)",
     "(u & 0x80000000u) ? u : (u | 0x80000000u)"),
    ("tie_to_higher_index", "return x->idx < y->idx ? -1 : 1;", "return x->idx > y->idx ? -1 : 1;"),
    ("keys_ascending", "return x->key > y->key ? -1 : 1;", "return x->key < y->key ? -1 : 1;"),
    ("block_max_reads_tail", "int64_t c1 = c0 + B < ec ? c0 + B : ec;",
     "int64_t c1 = c0 + B < W ? c0 + B : W;"),
    ("pin_from_clamped_end", "c[Kb] = (int32_t)oracle_pin(s, e, B);",
     "c[Kb] = (int32_t)oracle_pin(s, e < W ? e : W, B);"),
    ("edge_dropped", "edge = 1; /* clamped to the last column */", "edge = 0;"),
    ("mask_full_width", "for (int64_t c = 0; c < ec; ++c) {\n    int keep = 0;",
     "for (int64_t c = 0; c < W; ++c) {\n    int keep = 0;"),
    ("mask_spares_before_start", "    int keep = 0;\n    if (c >= s)",
     "    int keep = c < s;\n    if (c >= s)"),
    ("partial_block_dropped", "return (ec - s + B - 1) / B;", "return (ec - s) / B;"),
    ("topk_unsorted", "qsort(cols, (size_t)take, sizeof(int64_t), ascending_i64);", ""),
    ("block_topk_one_short", "int64_t take = NB < Kb ? NB : Kb;",
     "int64_t take = NB < Kb ? NB : Kb - 1;"),
    ("causal_offset_wrong", "if (causal) e = e - (rep - 1) + (r % rep);",
     "if (causal) e = e + (r % rep);"),
    ("edge_wrong_column", "(c == W - 1 && edge)", "(c == W - 2 && edge)"),
    ("packed_column_ignores_start", "if (s + b * (int64_t)B < W)", "if (b * (int64_t)B < W)"),
    ("row_topk_take_one_short", "int64_t take = L < K ? L : K;", "int64_t take = L < K ? L : K - 1;"),
    ("window_one_short", "int64_t w0 = w1 - window > s ? w1 - window : s;",
     "int64_t w0 = w1 - window + 1 > s ? w1 - window + 1 : s;"),
    ("combine_keeps_duplicates", "if (m == 0 || all[i] != all[m - 1]) all[m++] = all[i];",
     "all[m++] = all[i];"),
    ("attention_counts_instead_of_weights", "        l += p;\n", "        l += 1.0;\n"),
    ("lse_without_max", "lse[(int64_t)t * H + h] = m + log(l);", "lse[(int64_t)t * H + h] = log(l);"),
    ("union_mask_absolute_bit", "mask[p] |= 1u << (t - t0);", "mask[p] |= 1u << t;"),
    ("bf16_wrong_shift", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    ("score_without_scale", "s[i] = scale * dot;", "s[i] = dot;"),
    ("union_drops_last_token", "int32_t t1 = t0 + G < T ? t0 + G : T;",
     "int32_t t1 = t0 + G - 1 < T ? t0 + G - 1 : T;"),
]


def _pins_fail(orc) -> list:
    failed = []
    checks = [("golden:" + c["name"], lambda c=c: pins.test_hand_worked_rows(orc, c))
              for c in load_golden()["cases"]]
    checks += [
        ("combine_hand", lambda: combine.test_hand_worked(orc)),
        ("combine_span", lambda: combine.test_full_window_is_the_span(orc)),
        ("combine_union", lambda: combine.test_set_union_on_random_rows(orc)),
        ("block_scores", lambda: pins.test_hand_worked_block_scores(orc)),
        ("key_order", lambda: pins.test_key_is_total_order(orc)),
        ("brute", lambda: pins.test_brute_force_tiny(orc, False)),
        ("brute_exotic", lambda: pins.test_brute_force_tiny(orc, True)),
        ("brute_repeat", lambda: pins.test_brute_force_row_repeat(orc)),
        ("b1_reduction", lambda: pins.test_b1_reduces_to_stable_topk(orc)),
        ("invariants", lambda: pins.test_invariants_and_idempotence_random(orc)),
        ("att_bf16", lambda: att.test_bf16_decoding(orc)),
        ("att_single", lambda: att.test_single_position_is_that_row(orc)),
        ("att_equal", lambda: att.test_equal_scores_average_the_values(orc)),
        ("att_numpy", lambda: att.test_matches_an_independent_numpy_softmax(orc)),
        ("att_order", lambda: att.test_order_and_padding_do_not_matter(orc)),
        ("att_empty", lambda: att.test_empty_selection(orc)),
        ("att_union", lambda: att.test_union_against_sets(orc)),
    ]
    for name, fn in checks:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_mutant_table_matches_source():
    src = open(oracle.SOURCE).read()
    for name, find, _ in MUTANTS:
        assert src.count(find) == 1, f"mutant {name}: its target text must occur once"


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_each_mutant_is_caught(tmp_path, name, find, repl):
    src = open(oracle.SOURCE).read()
    assert src.count(find) == 1
    mutated = tmp_path / f"{name}.c"
    mutated.write_text(src.replace(find, repl))
    so = oracle.compile_oracle(str(mutated), str(tmp_path / f"lib{name}.so"))
    failed = _pins_fail(oracle.Oracle(so))
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path):
    so = oracle.compile_oracle(oracle.SOURCE, str(tmp_path / "libcopy.so"))
    assert _pins_fail(oracle.Oracle(so)) == []
