"""The oracle's pins catch plausible mistakes: each case plants one mistake in a copy of
moe_oracle.c (a misplaced reset, a transposed index, an off-by-one, a wrong rounding, a
weight paired with the wrong expert, ...), builds it, and runs the pins that should notice
it against that build. Every pin must fail on its mutant. The planted mistakes keep every
index inside its array, so a mutant computes wrong values but never writes out of bounds.
CPU only; the real oracle is untouched."""
import functools
import os

import pytest

import oracle
import workloads
from tests import test_oracle_layout as lay_pins
from tests import test_oracle_numerics as num_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

SMALL = num_pins.SMALL

# (name, original text, planted mistake, pins that must fail)
MUTATIONS = [
    ("eoff-inclusive-scan",
     "eoff[((int64_t)d * L + l) * N + s] = run;\n                run += cnt[(int64_t)s * E + e];",
     "run += cnt[(int64_t)s * E + e];\n                eoff[((int64_t)d * L + l) * N + s] = run;",
     [lay_pins.test_layout_matches_bruteforce_on_tiny_config]),
    ("ranks-reset-per-token",
     "int32_t rk = running[e]++;",
     "if (k == 0) memset(running, 0, sizeof(int32_t) * (size_t)E);\n                int32_t rk = running[e]++;",
     [lay_pins.test_layout_matches_bruteforce_on_tiny_config]),
    ("wrong-local-expert",
     "int d = e / L, l = e % L;",
     "int d = e / L, l = (e + 1) % L;",
     [lay_pins.test_layout_matches_bruteforce_on_tiny_config]),
    ("roff-scans-transposed-C",
     "roff[d * N + s] = run;\n            run += C[s * N + d];",
     "roff[d * N + s] = run;\n            run += C[d * N + s];",
     [lay_pins.test_layout_matches_bruteforce_on_random_tiny_shapes]),
    ("capacity-one-short",
     "if (sl < cap) {",
     "if (sl < cap - 1) {",
     [lay_pins.test_layout_matches_bruteforce_on_random_tiny_shapes]),
    ("e4m3-ties-away-from-zero",
     "return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;",
     "return f + 1.0;",
     [num_pins.test_e4m3_encode_matches_exhaustive_nearest]),
    ("fp8-scale-divisor",
     "float scale = (amax == 0.0f) ? 1.0f : amax / 448.0f;",
     "float scale = (amax == 0.0f) ? 1.0f : amax / 447.0f;",
     [num_pins.test_quantize_fp8_scale_and_bound]),
    ("dequant-divides",
     "float y = qv * sc;",
     "float y = qv / sc;",
     [num_pins.test_expert_dequant_definition]),
    ("dispatch-recv-off-by-one",
     "int64_t src0 = roff[d * N + s] + soff[(int64_t)s * E + e] - soff[(int64_t)s * E + d * L];\n"
     "                int64_t dst0 = eoff[((int64_t)d * L + l) * N + s];",
     "int64_t src0 = roff[d * N + s] + soff[(int64_t)s * E + e] - soff[(int64_t)s * E + d * L] + 1;\n"
     "                int64_t dst0 = eoff[((int64_t)d * L + l) * N + s];",
     [functools.partial(num_pins.test_payload_rows_are_the_routed_tokens, wl=SMALL[1])]),
    ("combine-send-slice-of-wrong-expert",
     "memcpy(crecv + ((int64_t)s * TR + soff[(int64_t)s * E + d * L]) * H,",
     "memcpy(crecv + ((int64_t)s * TR + soff[(int64_t)s * E + d]) * H,",
     [functools.partial(num_pins.test_round_trip_exact_with_equal_power_of_two_weights, R=4)]),
    ("combine-weight-of-next-slot",
     "float prod = w[q] * y;",
     "float prod = w[q - k + (k + 1) % R] * y;",
     [functools.partial(num_pins.test_combine_with_distinct_expert_outputs_restated, wl=num_pins.DISTINCT[0])]),
    ("combine-keeps-dropped-pairs",
     "if (pos[q] < 0 || slot[q] < 0) continue;",
     "if (pos[q] < 0) continue;",
     [num_pins.test_combine_skips_dropped_and_invalid_pairs]),
    ("partial-groups-descending",
     "int j = 0;\n            for (int d = 0; d < N; d++) {",
     "int j = 0;\n            for (int d = N - 1; d >= 0; d--) {",
     [functools.partial(num_pins.test_partial_combine_with_distinct_expert_outputs_restated,
                        wl=num_pins.DISTINCT[0])]),
]


@pytest.mark.parametrize("name,orig,mutant,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(orc, tmp_path, name, orig, mutant, pins):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"{name}: mutation site not found exactly once"
    path = tmp_path / "moe_oracle_mutant.c"
    path.write_text(src.replace(orig, mutant))
    so = oracle.compile_source(str(path), str(tmp_path / f"libmoe_oracle_{name}.so"))
    for pin in pins:
        pin(orc)                                   # the real oracle passes the pin ...
        with oracle.library(so):
            with pytest.raises((AssertionError, IndexError, ValueError)):
                pin(orc)                           # ... and the mutant fails it
