"""Planted mistakes in the KPool part of the oracle: each mutant must fail a pin.

A mutant is a copy of oracle/csa_oracle.cpp with one plausible KPool mistake (the pool
grid ignoring the first valid key, a dropped last pool, the gate of the wrong key, keys
in reverse order, a weight or a product not cast to bf16 under compression, an error
mass without its exponent term or set to zero, a slack that never or always fires),
compiled to a temporary library on the CPU. The pins re-run against it are the
brute-force evaluator, the hand-derived examples, the float32 evaluation and the slack
sweep of test_kpool_oracle.py. No mutant reads outside its buffers.
"""
import os

import pytest

import oracle
from tests.test_kpool_oracle import kpool_pin_failures

SRC = os.path.join(os.path.dirname(oracle.__file__), "csa_oracle.cpp")

MUTANTS = {
    "pool_grid_ignores_lead": (
        "const int64_t first = static_cast<int64_t>(cu[s]) + (lead != nullptr ? lead[s] : 0);",
        "const int64_t first = static_cast<int64_t>(cu[s]);"),
    "last_pool_dropped": (
        "const int64_t n = valid > 0 ? valid / P : 0;",
        "const int64_t n = valid > 0 ? valid / P - (valid >= 2 * P ? 1 : 0) : 0;"),
    "gate_of_first_key": (
        "x[i] = bf16_bits_to_double(gate[flat]);",
        "x[i] = bf16_bits_to_double(gate[start * d + j]);"),
    "keys_reversed": (
        "v[i] = bf16_bits_to_double(key[flat]);",
        "v[i] = bf16_bits_to_double(key[(start + P - 1 - i) * d + j]);"),
    "weight_not_cast_to_bf16": (
        "const double pb = bf16_bits_to_double(double_to_bf16_bits(pf));         // cast to bf16",
        "const double pb = pf;"),
    "product_not_cast_to_bf16": (
        "const double prod = bf16_bits_to_double(double_to_bf16_bits(pb * v[i]));  // bf16 product",
        "const double prod = pb * v[i];"),
    "mass_without_exponent_term": (
        "r.err += p[i] * (std::fabs(v[i]) + std::fabs(v[i] - r.o) * (1.0 + std::fabs(x[i]) + std::fabs(m)));",
        "r.err += p[i] * (std::fabs(v[i]) + std::fabs(v[i] - r.o));"),
    "compression_mass_zero": ("r.err = P * abs_sum;", "r.err = 0.0 * abs_sum;"),
    "slack_never": ("r.slack += worst;", "r.slack += 0.0 * worst;"),
    "slack_always": (
        "if (qb != pb) worst = std::max(worst, std::fabs(alt - prod));",
        "worst = std::max(worst, std::fabs(alt - prod) + 1e-3);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_kpool_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mut = tmp_path / "mutant.cpp"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    oracle.build(force=True, src=str(mut), out=str(so))
    lib = oracle.load(str(so))
    assert kpool_pin_failures(lib), f"mutant {name} passed every pin"
