"""Planted mistakes in the oracle must be caught by the pins.

Each mutant is a copy of the oracle's C source with one plausible mistake (a
dropped term, a wrong sign, a wrong operand, a wrong order), compiled on the
CPU into a temporary directory.  The test passes only if at least one pin in
``tests/oracle_pins.py`` fails on that build -- evidence that the pins would
notice the same mistake in the committed oracle.
"""
import os

import pytest

import oracle
from oracle import build as obuild
from tests import oracle_pins

# (name, text in the source, replacement, occurrences expected)
MUTANTS = [
    ("mean_square_becomes_sum",
     "logit[i] = sd / sqrt(s2 / (double)H + j->eps);",
     "logit[i] = sd / sqrt(s2 + j->eps);", 1),
    ("eps_outside_sqrt",
     "logit[i] = sd / sqrt(s2 / (double)H + j->eps);",
     "logit[i] = sd / (sqrt(s2 / (double)H) + j->eps);", 1),
    ("sum_of_squares_drops_square",
     "s2 += v * v;", "s2 += v;", 1),
    ("softmax_sign_flipped",
     "w[i] = exp(logit[i] - m);", "w[i] = exp(m - logit[i]);", 1),
    ("softmax_without_max_shift",
     "w[i] = exp(logit[i] - m);", "w[i] = exp(logit[i]);", 1),
    ("mix_normalised_rows",
     "acc[h] += w[i] * bf16_to_double(x[h]);",
     "acc[h] += w[i] * bf16_to_double(x[h]) / sqrt(ss[i] / (double)H + j->eps);", 1),
    ("query_drops_res_w",
     "q[h] = bf16_to_double(rms_w[h]) * bf16_to_double(res_w[h]);",
     "q[h] = bf16_to_double(rms_w[h]);", 1),
    ("current_row_ignores_delta",
     "                : c;", "                : prow;", 2),
    ("bank_slots_reversed",
     "(int64_t)i * j->blocks_slot", "(int64_t)(S - 1 - i) * j->blocks_slot", 2),
    ("writeback_stores_output",
     "memcpy(dst, c, (size_t)H * sizeof(uint16_t));",
     "memcpy(dst, orow, (size_t)H * sizeof(uint16_t));", 1),
    ("output_norm_drops_weight",
     "orow[h] = double_to_bf16_rne(acc[h] * r * bf16_to_double(j->out_norm_w[h]));",
     "orow[h] = double_to_bf16_rne(acc[h] * r);", 1),
    ("output_norm_uses_eps",
     "sq / (double)H + j->out_eps", "sq / (double)H + j->eps", 1),
    ("rounding_ties_away",
     "if (frac > 0.5 || (frac == 0.5 && (n & 1u))) n += 1u;",
     "if (frac >= 0.5) n += 1u;", 1),
    ("rounding_truncates",
     "if (frac > 0.5 || (frac == 0.5 && (n & 1u))) n += 1u;", "", 1),
    ("grouped_bank_row_modulo",
     "j->blocks + (t / j->group) * j->blocks_token : NULL;",
     "j->blocks + (t % j->group) * j->blocks_token : NULL;", 1),
    ("grouped_first_row_writes",
     "(t % j->group == j->group - 1 || t == j->T - 1)", "(t % j->group == 0)", 1),
    ("grouped_write_into_source_accepted",
     "if (blocks_group > 1 && block_write_idx >= 0 && block_write_idx < num_blocks)",
     "if (0)", 1),
    ("writeback_before_reads",
     "  /* steps 2-4: per-candidate sum of squares, dot with q, logit */",
     "  if (j->block_write_idx >= 0)\n"
     "    memcpy(j->blocks + t * j->blocks_token + (int64_t)j->block_write_idx * j->blocks_slot,\n"
     "           c, (size_t)H * sizeof(uint16_t));", 1),
]


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, count):
    with open(obuild.SRC) as f:
        src = f.read()
    assert src.count(old) == count, f"mutation site for {name} moved"
    mutated = src.replace(old, new)
    path = os.path.join(tmp_path, f"{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = obuild.compile_source(path, os.path.join(tmp_path, f"lib{name}.so"))
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
            break
        except (ValueError, FloatingPointError, OverflowError):
            caught.append(pin.__name__)
            break
    assert caught, f"no pin notices the planted mistake {name}"
