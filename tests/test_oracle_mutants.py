"""Mutation check of the oracle pins (CPU only).

Each case plants one plausible mistake in a copy of the oracle's C source,
builds it, and runs the pins against the mutant.  Every mutant must make at
least one pin fail; a mutant that survives would mean the pins cannot see
that kind of mistake.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sse_oracle.c")

MUTANTS = {
    "selected_state_not_decayed": ("a[r] * Si[(size_t)r * d + col] + e[i] * kk[r] * v[col]",
                                   "Si[(size_t)r * d + col] + e[i] * kk[r] * v[col]"),
    "write_decayed_too": ("a[r] * Si[(size_t)r * d + col] + e[i] * kk[r] * v[col]",
                          "a[r] * (Si[(size_t)r * d + col] + e[i] * kk[r] * v[col])"),
    "write_without_router_weight": ("a[r] * Si[(size_t)r * d + col] + e[i] * kk[r] * v[col]",
                                    "a[r] * Si[(size_t)r * d + col] + kk[r] * v[col]"),
    "read_without_router_weight": ("const double w = e[i] * D->scale * q[r];",
                                   "const double w = D->scale * q[r];"),
    "ties_to_higher_index": ("logit[i] > logit[best]", "logit[i] >= logit[best]"),
    "shared_not_decayed": ("a[r] * Sn[(size_t)r * d + col] + ks[r] * v[col]",
                           "Sn[(size_t)r * d + col] + ks[r] * v[col]"),
    "gate_sign_flipped": ("a[r] = exp(g[r]);", "a[r] = exp(-g[r]);"),
    "softmax_not_normalised": ("e[i] /= s;", "(void)s;"),
    "shared_key_from_query": ("k_shared ? k_shared : kk", "k_shared ? k_shared : q"),
    "read_columns_reversed": ("out[col] += w * Si[(size_t)r * d + col];",
                              "out[col] += w * Si[(size_t)r * d + (d - 1 - col)];"),
    "gate_row_index_wrong": ("a[r] = exp(g[r]);", "a[r] = exp(g[c - 1 - r]);"),
}

PIN_FUNCS = [
    pins.test_textbook_linear_attention,
    lambda: pins.test_recurrence_matches_unrolled_closed_form(2, 1, False),
    lambda: pins.test_recurrence_matches_unrolled_closed_form(1, 1, True),
    pins.test_equal_logits_all_selected_is_scaled_dense_gla,
    pins.test_local_update_clock_worked_example,
    pins.test_routing_matches_stable_argsort_and_weights_not_renormalised,
    pins.test_unselected_partitions_bitwise_unchanged,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_killed(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, "anchor text not found; update the mutant"
    mutated = src.replace(old, new)
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "mutant.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so_path),
                    str(c_path), "-lm"], check=True)
    failures = 0
    with oracle._library_override(str(so_path)):
        for f in PIN_FUNCS:
            try:
                f()
            except AssertionError:
                failures += 1
    assert failures > 0, f"mutant {name} survived every pin"
