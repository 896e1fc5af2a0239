"""Planted mistakes: each mutant of the oracle source must fail at least one pin.

A mutant is a copy of oracle/csa_oracle.cpp with one plausible mistake (a swapped
half, a reversed ape row, a dropped term, a flipped sign, an off-by-one mask, an error
mass of the parity tolerance shrunk or inflated),
compiled to a temporary library on the CPU. The pins re-run against it are the
brute-force evaluator, the hand-derived golden pack (values and error masses) and
the softmax identities from test_oracle_pins.py. No mutant reads outside its buffers.
"""
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import thd_synth as ts
from tests.test_oracle_pins import GOLDEN, brute_force, golden_mass_mismatches, tiny_packs

SRC = os.path.join(os.path.dirname(oracle.__file__), "csa_oracle.cpp")

MUTANTS = {
    "prev_half_reads_own_columns": (
        "win.push_back({t, j, static_cast<int64_t>(w) * C + j});\n    }\n  }",
        "win.push_back({t, d + j, static_cast<int64_t>(w) * C + j});\n    }\n  }"),
    "own_half_reads_first_columns": (
        "win.push_back({t, d + j, static_cast<int64_t>(w) * C + d + j});",
        "win.push_back({t, j, static_cast<int64_t>(w) * C + d + j});"),
    "ape_row_reversed": (
        "win.push_back({t, d + j, static_cast<int64_t>(w) * C + d + j});",
        "win.push_back({t, d + j, static_cast<int64_t>(ratio - 1 - w) * C + d + j});"),
    "ape_dropped": (
        "bf16_bits_to_double(score[flat]) + static_cast<double>(ape[win[i].ape_index]);",
        "bf16_bits_to_double(score[flat]) + 0.0;"),
    "dscore_sign_flipped": (
        "const double ds = st.p[i] * g * (st.v[i] - st.o);",
        "const double ds = st.p[i] * g * (st.o - st.v[i]);"),
    "first_two_blocks_masked": ("if (b >= 1) {", "if (b >= 2) {"),
    "softmax_not_normalised": ("for (size_t i = 0; i < n; ++i) st.p[i] /= z;", ""),
    "max_not_subtracted_and_first_only": (
        "st.p[i] = std::exp(st.x[i] - st.m);", "st.p[i] = std::exp(st.x[i] - st.x[0]) * (i == 0 ? 2.0 : 1.0);"),
    "dape_sums_dkv": ("my_dape[win[i].ape_index] += ds;", "my_dape[win[i].ape_index] += dk;"),
    "score_grad_uses_kv_only": (
        "gsc[flat] = ds;", "gsc[flat] = dk;"),
    # the parity tolerance's error masses: each shrunk or inflated mass must fail a pin
    "out_err_without_exponent_term": (
        "std::fabs(st.v[i] - st.o) * (1.0 + std::fabs(st.x[i]) + std::fabs(st.m)));",
        "std::fabs(st.v[i] - st.o));"),
    "out_err_doubled": ("  return a;\n}", "  return 2.0 * a;\n}"),
    "dkv_err_without_exponent_term": (
        "gkv_err[flat] = std::fabs(dk) * xm;", "gkv_err[flat] = std::fabs(dk);"),
    "dscore_err_without_out_err": (
        "(std::fabs(st.v[i] - st.o) * xm + oerr)", "(std::fabs(st.v[i] - st.o) * xm)"),
    "dape_err_without_abs": (
        "my_err[win[i].ape_index] += err + std::fabs(ds);", "my_err[win[i].ape_index] += err;"),
}


def _run_pins(lib):
    """Returns the list of pin names that fail for ``lib``."""
    failed = []
    for k, pack in enumerate(tiny_packs()[:3]):
        bf = brute_force(pack)
        try:
            f = oracle.fwd_pack(pack, want_f64=True, lib=lib)
            b = oracle.bwd_pack(pack, want_f64=True, want_owners=True, lib=lib)
        except oracle.OracleError:
            failed.append(f"error{k}")
            continue
        if not np.allclose(f["out_f64"], bf["out"], rtol=1e-13, atol=1e-15):
            failed.append(f"fwd{k}")
        if not (b["owners"] == bf["owners"]).all():
            failed.append(f"owners{k}")
        for key, ref in (("dkv_f64", "dkv"), ("dscore_f64", "dscore"), ("dape_f64", "dape")):
            if not np.allclose(b[key], bf[ref], rtol=1e-12, atol=1e-14):
                failed.append(f"{key}{k}")
    with open(os.path.join(GOLDEN, "hand_pack_r2_c2.json")) as fh:
        gd = json.load(fh)
    env = {"e": math.e, "__builtins__": {}}
    kv = ts.f32_to_bf16_bits(np.array(gd["kv"], np.float32))
    score = ts.f32_to_bf16_bits(np.array(gd["score"], np.float32))
    f = oracle.fwd(kv, score, np.array(gd["ape"], np.float32), np.array(gd["cu_seqlens"], np.int32),
                   2, 2, 1, 7, want_f64=True, lib=lib)
    if not np.allclose(f["out_f64"][:, 0], [eval(s, env) for s in gd["expected"]["out"]],
                       rtol=1e-15):
        failed.append("golden")
    failed += ["golden_" + m for m in golden_mass_mismatches(lib)]
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, oracle_lib):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mut = tmp_path / "mutant.cpp"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    oracle.build(force=True, src=str(mut), out=str(so))
    lib = oracle.load(str(so))
    assert _run_pins(lib), f"mutant {name} passed every pin"


def test_unmutated_oracle_passes(oracle_lib):
    assert _run_pins(oracle.load()) == []
