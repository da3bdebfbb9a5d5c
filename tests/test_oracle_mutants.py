"""Mutation check of the oracle pins (no GPU).

Each case compiles a copy of oracle/gdn_oracle.c with one plausible mistake
planted in it (on the CPU, in a temporary directory) and asserts that at least
one pin of test_oracle_pins.py fails against the mutant.  This shows the pins
would catch that class of slip in the oracle itself.
"""
import os
import subprocess

import pytest

import test_oracle_pins as pins
from oracle import oracle as oracle_pkg

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "gdn_oracle.c")

MUTANTS = {
    "recurrence_drops_decay": ("S[(int64_t)d * V + e] = a * proj + b * kt[d] * vt[e];",
                               "S[(int64_t)d * V + e] = proj + b * kt[d] * vt[e];"),
    "recurrence_sign_flip": ("const double proj = S[(int64_t)d * V + e] - b * kt[d] * ktS[e];",
                             "const double proj = S[(int64_t)d * V + e] + b * kt[d] * ktS[e];"),
    "gqa_tiled_heads": ("const int hq = h / (Hv / Hqk);", "const int hq = h % Hqk;"),
    "output_before_update": ("for (int d = 0; d < K; ++d) acc += S[(int64_t)d * V + e] * qt[d];",
                             "for (int d = 0; d < K; ++d) acc += (S[(int64_t)d * V + e] - kt[d] * b * (vt[e] - a * ktS[e])) / a * qt[d];"),
    "chunk_o_strict_mask": ("if (j <= i) {", "if (j < i) {"),
    "chunk_h_wrong_glast": ("const double glast = sc->gamma[n - 1];", "const double glast = sc->gamma[0];"),
    "wy_beta_on_rows": ("a += sc->T[i * n + c] * BV(c) * VR(c)[e];", "a += sc->T[i * n + c] * BV(i) * VR(c)[e];"),
    "chunk_o_no_decay_on_state": ("oi[e] = scale * (exp(sc->gamma[i]) * inter + intra);",
                                  "oi[e] = scale * (inter + intra);"),
    "kkt_missing_beta": ("a = BV(i) * exp(sc->gamma[i] - sc->gamma[j]) * dot;",
                         "a = exp(sc->gamma[i] - sc->gamma[j]) * dot;"),
}

# pin checks that take an oracle object exposing recurrent() / chunked()
CHECKS = [
    lambda o: [pins.test_hand_worked_examples(o, c, f) for c in pins._golden_cases()
               for f in ("recurrent", "chunked_C1", "chunked_C2")],
    lambda o: pins.test_chunked_equals_recurrent(o, 16, 0),
    lambda o: pins.test_chunked_equals_recurrent(o, 64, 1),
    lambda o: pins.test_beta_zero_is_pure_decay(o, "recurrent"),
    lambda o: pins.test_delta_rule_overwrite_orthonormal_keys(o, "recurrent"),
    lambda o: pins.test_householder_reflection_preserves_state(o, "recurrent"),
    lambda o: pins.test_fixed_point_when_values_match_predictions(o, "recurrent"),
    lambda o: pins.test_gqa_maps_value_head_to_group(o),
    lambda o: pins.test_output_uses_post_update_state(o),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old}"
    mpath = tmp_path / f"{name}.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(mpath), "-o", str(so), "-lm"],
                   check=True)
    mutant = oracle_pkg.Oracle(str(so))
    failures = 0
    for check in CHECKS:
        try:
            check(mutant)
        except AssertionError:
            failures += 1
    assert failures >= 1, f"no pin caught mutant {name}"
