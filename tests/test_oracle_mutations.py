"""Mutation tests: each plants one plausible mistake in a copy of the oracle's
C source (on the CPU, in a temporary directory), builds it, and checks that at
least one of the oracle pins fails.  A pin set that let a mutant through would
not be pinning that part of the oracle.

The first two mutants are the defects the simulator page's "Negative-tested"
table names (packing shift 8 -> 7; shared gate multiply dropped)."""
import os

import pytest

import test_oracle_pins as pins
from oracle import oracle as O

SRC = os.path.join(os.path.dirname(O.__file__), "moe_oracle.c")

# (name, original text, mutated text, pins expected to catch it)
MUTANTS = [
    ("pack shift 8 -> 7", "((uint32_t)num_experts << 8)", "((uint32_t)num_experts << 7)",
     [pins.check_shape_words]),
    ("shared gate multiply dropped", "double g = c->gate ? c->gate[i] : 1.0;",
     "double g = 1.0;", [pins.check_gate, pins.check_dense_masked_form]),
    ("ties to the higher index", "if (best < 0 || l[e] > l[best])",
     "if (best < 0 || l[e] >= l[best])", [pins.check_topk_bruteforce,
                                          pins.check_topk_wide_blocks]),
    ("renormalised weights everywhere", "if (norm_topk) {", "if (1) {",
     [pins.check_topk_bruteforce, pins.check_dense_masked_form]),
    ("silu sign", "a_scratch[j] = g / (1.0 + exp(-g)) * u;",
     "a_scratch[j] = g / (1.0 + exp(g)) * u;",
     [pins.check_single_expert_textbook, pins.check_dense_masked_form]),
    ("down weight transposed", "o += a_scratch[j] * ld(wd, wdt, h * I + j);",
     "o += a_scratch[j] * ld(wd, wdt, j * H + h);", [pins.check_single_expert_textbook]),
    ("gate and up swapped", "a_scratch[j] = g / (1.0 + exp(-g)) * u;",
     "a_scratch[j] = u / (1.0 + exp(-u)) * g;", [pins.check_single_expert_textbook]),
    ("route weight dropped", "c->w[i * c->k + s], a, yr);", "1.0, a, yr);",
     [pins.check_combine_is_k_sum, pins.check_all_duplicate_closed_form]),
    ("only first slot combined", "for (int32_t s = 0; s < c->k; s++) {\n      int64_t e",
     "for (int32_t s = 0; s < 1; s++) {\n      int64_t e",
     [pins.check_combine_is_k_sum, pins.check_all_duplicate_closed_form]),
    ("group rows in reverse", "int32_t r = next[e]++;",
     "int32_t r = offsets[e + 1] - 1 - (next[e]++ - offsets[e]);",
     [pins.check_permute_bruteforce]),
    ("offsets off by one expert", "offsets[e + 1] = offsets[e] + counts[e];",
     "offsets[e + 1] = offsets[e] + (e > 0 ? counts[e - 1] : counts[e]);",
     [pins.check_permute_bruteforce]),
    ("expert stride ignored for up", "base_u + e * c->su * esz",
     "base_u + e * c->sg * esz", [pins.check_expert_strides_and_tokens]),
    ("router row index", "ld(c->wr, c->wdt, col * c->H + h)",
     "ld(c->wr, c->wdt, h * c->ncols + col)", [pins.check_dense_masked_form]),
    ("sigmoid sign", "gate[t] = 1.0 / (1.0 + exp(-z[t * ld_z]));",
     "gate[t] = 1.0 / (1.0 + exp(z[t * ld_z]));", [pins.check_gate]),
    ("rmsnorm eps dropped", "1.0 / sqrt(ss / (double)H + eps)", "1.0 / sqrt(ss / (double)H)",
     [pins.check_rmsnorm_closed_forms, pins.check_rmsnorm_high_precision]),
    ("rmsnorm mean of x, not x^2", "ss += v * v;", "ss += fabs(v);",
     [pins.check_rmsnorm_closed_forms, pins.check_rmsnorm_high_precision]),
    ("norm weight ignored", "* inv * ld(w, dtype, h)", "* inv",
     [pins.check_rmsnorm_closed_forms]),
    ("rounding truncates", "r = rint(a / q) * q;", "r = floor(a / q) * q;",
     [pins.check_round_act, pins.check_rmsnorm_high_precision]),
    ("rounding keeps 7 bits", "q = ldexp(1.0, e - 8);", "q = ldexp(1.0, e - 7);",
     [pins.check_round_act]),
]


@pytest.mark.parametrize("name,orig,mut,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, orc, name, orig, mut, checks):
    src = open(SRC).read()
    assert src.count(orig) == 1, "mutation site not unique: %r" % orig
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(orig, mut))
    so = O.build(force=True, src=str(msrc), out=str(tmp_path / "mutant.so"))
    saved = O._lib
    O._lib = O.load(so)
    try:
        caught = []
        for chk in checks:
            try:
                chk()
            except (AssertionError, ValueError):
                caught.append(chk.__name__)
        assert caught, "mutant %r passed every pin" % name
    finally:
        O._lib = saved
