"""Pins for the KPool part of the fp64 oracle, independent of the oracle's own code (CPU).

KPool is the DSA indexer's key pooling ("Megatron-LM PR #8835", the KPool commits): an
FP32 softmax of a gate over pools of P consecutive keys, the pool grid starting at each
segment's first valid key, and, with key-dtype compression, the softmax cast to bf16
before multiplying and reducing. Each test checks the oracle against something it cannot
share a mistake with:

* a brute-force evaluator that finds each pool's members by scanning every token of the
  pack against a membership predicate (Python floats, math.exp, math.fsum), not the
  oracle's pool list;
* the pool count, counted here by scanning tokens for pool starts;
* invariants: equal gates give the pool mean, a common gate shift changes nothing,
  P = 1 is the identity in both modes, a segment's lead equals dropping its first keys,
  and with no leads the FP32 mode is the compressor's coff=1 forward with ape = 0;
* hand-derived examples (tests/golden/kpool_hand.json), values, bits and an error mass;
* a plain float32 evaluation of every pool lands within ulp + 8 u32 mass (+ slack);
* the slack is non-zero exactly where a weight sits within its evaluation window of a
  bf16 rounding boundary.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import thd_synth as ts

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U32 = 2.0 ** -24
KAPPA = 8.0


def _vals(bits):
    return ts.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


def _bf16(x):
    """bf16 round-to-nearest-even of doubles, through the oracle's rounding (pinned by a
    brute-force nearest search in test_oracle_pins.py)."""
    return oracle.round_bf16(np.asarray(x, dtype=np.float64))


# ----------------------------------------------------------------------------------
# Independent brute-force evaluator (predicate formulation)
# ----------------------------------------------------------------------------------

def brute_pools(cu, lead, P):
    """Pool starts in token order, found by scanning: a token starts a pool when it lies
    at or after its segment's first valid key, its offset from that key is a multiple of
    P, and P keys of the segment follow from it (itself included)."""
    S = len(cu) - 1
    starts = []
    for t in range(int(cu[0]), int(cu[S]) if S else 0):
        s = max(i for i in range(S) if cu[i] <= t < cu[i + 1])
        first = cu[s] + (0 if lead is None else int(lead[s]))
        if t >= first and (t - first) % P == 0 and t + P <= cu[s + 1]:
            starts.append(t)
    return starts


def brute_kpool(pack, compress=False):
    cu = [int(x) for x in pack.cu_seqlens]
    key, gate = _vals(pack.key), _vals(pack.gate)
    P, d = pack.pool, pack.d
    starts = brute_pools(cu, pack.lead, P)
    out = np.zeros((len(starts), d))
    for o, t0 in enumerate(starts):
        for j in range(d):
            x = [float(gate[t0 + i, j]) for i in range(P)]
            v = [float(key[t0 + i, j]) for i in range(P)]
            m = max(x)
            e = [math.exp(xi - m) for xi in x]
            z = math.fsum(e)
            p = [ei / z for ei in e]
            if not compress:
                out[o, j] = math.fsum(pi * vi for pi, vi in zip(p, v))
            else:
                pf = np.float32(p).astype(np.float64)               # FP32 weights
                pb = _vals(ts.f32_to_bf16_bits(pf.astype(np.float32)))  # cast to bf16
                prod = _bf16(pb * np.array(v))                      # bf16 products
                out[o, j] = math.fsum(float(q) for q in _vals(prod))
    return out, starts


def kpool_tiny_packs():
    return [
        ts.make_kpool("kpool_tiny"),
        ts.make_kpool_custom([7, 1, 0, 12, 6], pool=3, d=5, leads=[2, 0, 0, 1, 7], pad_rows=3,
                             seed=11),
        ts.make_kpool_custom([9, 8], pool=2, d=3, seed=12, gate_scale=4.0),
        ts.make_kpool_custom([16, 5], pool=8, d=4, leads=[3, 0], seed=13),
        ts.make_kpool_custom([5], pool=1, d=6, leads=[2], pad_rows=2, seed=14),
    ]


@pytest.fixture(scope="module")
def oracle_lib():
    return oracle.load()


@pytest.mark.parametrize("k", range(5))
@pytest.mark.parametrize("compress", [False, True])
def test_kpool_matches_brute_force(oracle_lib, k, compress):
    pack = kpool_tiny_packs()[k]
    bf, starts = brute_kpool(pack, compress)
    r = oracle.kpool_fwd_pack(pack, compress=compress, want_f64=True)
    assert r["out"].shape == bf.shape
    np.testing.assert_allclose(r["out_f64"], bf, rtol=1e-13, atol=1e-15)
    assert (r["out"] == _bf16(bf)).all()


def test_kpool_total_matches_scan(oracle_lib):
    for pack in kpool_tiny_packs():
        _, starts = brute_pools_count(pack)
        assert oracle.kpool_total(pack.cu_seqlens, pack.lead, pack.pool) == len(starts)
        assert pack.total_pools == len(starts)


def brute_pools_count(pack):
    cu = [int(x) for x in pack.cu_seqlens]
    starts = brute_pools(cu, pack.lead, pack.pool)
    return len(starts), starts


def test_golden_examples(oracle_lib):
    with open(os.path.join(GOLDEN, "kpool_hand.json")) as fh:
        gd = json.load(fh)
    env = {"e": math.e, "__builtins__": {}}
    for ex in gd["examples"]:
        key = ts.f32_to_bf16_bits(np.array(ex["key"], np.float32))
        gate = ts.f32_to_bf16_bits(np.array(ex["gate"], np.float32))
        cu = np.array(ex["cu_seqlens"], np.int32)
        lead = None if ex["lead"] is None else np.array(ex["lead"], np.int32)
        for mode, want in ex["expected"].items():
            r = oracle.kpool_fwd(key, gate, cu, lead, ex["P"], ex["d"], int(cu[-1]),
                                 compress=mode == "compress", want_f64=True, want_err=True)
            vals = [float(Fraction(s)) if "e" not in s else eval(s, env) for s in want["out_f64"]]
            np.testing.assert_allclose(r["out_f64"].reshape(-1), vals, rtol=1e-15, atol=0,
                                       err_msg=f"{ex['name']} {mode}")
            if "out_bits" in want:
                assert list(r["out"].reshape(-1)) == want["out_bits"], (ex["name"], mode)
            if "out_err" in want:
                np.testing.assert_allclose(r["out_err"].reshape(-1),
                                           [eval(s, env) for s in want["out_err"]], rtol=1e-14)


def test_equal_gates_give_pool_mean(oracle_lib):
    pack = ts.make_kpool_custom([12, 9], pool=4, d=6, leads=[1, 0], seed=21)
    pack.gate[:] = ts.f32_to_bf16_bits(np.full(pack.gate.shape, 0.75, np.float32))
    r = oracle.kpool_fwd_pack(pack, want_f64=True)
    key = _vals(pack.key)
    _, starts = brute_pools_count(pack)
    want = np.stack([key[t:t + 4].mean(axis=0) for t in starts])
    np.testing.assert_allclose(r["out_f64"], want, rtol=1e-14, atol=1e-16)


def test_common_gate_shift_changes_nothing(oracle_lib):
    """Gates on a coarse grid (multiples of 1/8 in [-2, 2]) shifted by 1 stay exact in bf16."""
    pack = ts.make_kpool_custom([12, 9, 7], pool=3, d=5, leads=[0, 2, 1], seed=22)
    g = np.round(ts.bf16_bits_to_f32(pack.gate) * 8).clip(-16, 16) / 8
    pack.gate[:] = ts.f32_to_bf16_bits(g.astype(np.float32))
    a = oracle.kpool_fwd_pack(pack, want_f64=True)
    pack.gate[:] = ts.f32_to_bf16_bits((g + 1.0).astype(np.float32))
    b = oracle.kpool_fwd_pack(pack, want_f64=True)
    np.testing.assert_allclose(a["out_f64"], b["out_f64"], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("compress", [False, True])
def test_pool_of_one_is_identity(oracle_lib, compress):
    pack = ts.make_kpool_custom([5, 0, 7], pool=1, d=9, leads=[1, 0, 3], seed=23)
    r = oracle.kpool_fwd_pack(pack, compress=compress)
    rows = [t for s in range(pack.S) for t in range(pack.cu_seqlens[s] + pack.lead[s],
                                                     pack.cu_seqlens[s + 1])]
    assert (r["out"] == pack.key[rows]).all()


def test_lead_equals_dropping_first_keys(oracle_lib):
    """A segment with lead l pools like the same segment with its first l keys removed."""
    pack = ts.make_kpool_custom([14, 11], pool=4, d=6, leads=[3, 2], seed=24)
    a = oracle.kpool_fwd_pack(pack, want_f64=True)
    keep = np.r_[3:14, 14 + 2:25]
    cut = ts.KPoolPack("cut", 4, 6, len(keep), np.array([0, 11, 20], np.int32), None,
                       pack.key[keep].copy(), pack.gate[keep].copy())
    b = oracle.kpool_fwd_pack(cut, want_f64=True)
    assert (a["out"] == b["out"]).all()
    np.testing.assert_array_equal(a["out_f64"], b["out_f64"])


def test_no_lead_fp32_mode_is_compressor_coff1(oracle_lib):
    """With no leads, KPool's FP32 mode is the compressor's coff=1 forward with ratio = P,
    score = gate, kv = key and ape = 0 (the compressor oracle is pinned on its own)."""
    pack = ts.make_kpool_custom([13, 4, 0, 9, 22], pool=4, d=7, pad_rows=3, seed=25)
    a = oracle.kpool_fwd_pack(pack, want_f64=True, want_err=True)
    ape = np.zeros((4, 7), np.float32)
    c = oracle.fwd(pack.key, pack.gate, ape, pack.cu_seqlens, 4, 1, 7, pack.capacity,
                   want_f64=True, want_err=True)
    assert (a["out"] == c["out"]).all()
    np.testing.assert_allclose(a["out_f64"], c["out_f64"], rtol=1e-15, atol=0)
    np.testing.assert_allclose(a["out_err"], c["out_err"], rtol=1e-15, atol=0)


def test_kpool_rejects_bad_inputs(oracle_lib):
    pack = ts.make_kpool("kpool_tiny")
    with pytest.raises(oracle.OracleError):
        oracle.kpool_fwd(pack.key, pack.gate, pack.cu_seqlens, np.array([0, -1, 0, 0, 0, 0],
                         np.int32), 4, 8, pack.capacity)
    with pytest.raises(oracle.OracleError):
        oracle.kpool_fwd(pack.key, pack.gate, pack.cu_seqlens, pack.lead, 4, 8, pack.capacity,
                         out_rows=pack.total_pools - 1)
    with pytest.raises(oracle.OracleError):
        oracle.kpool_fwd(pack.key, pack.gate, np.array([0, 9, 5], np.int32), None, 4, 8, 44)


# ----------------------------------------------------------------------------------
# Error mass and slack
# ----------------------------------------------------------------------------------

def f32_kpool(pack, compress):
    """Every pool evaluated in plain float32 (numpy, one rounding per operation, base-2
    exponent, sums in pool order); membership from brute_pools. Returns the values before
    the final bf16 cast."""
    cu = [int(x) for x in pack.cu_seqlens]
    key = ts.bf16_bits_to_f32(pack.key)
    gate = ts.bf16_bits_to_f32(pack.gate)
    P, d = pack.pool, pack.d
    starts = brute_pools(cu, pack.lead, P)
    out = np.zeros((len(starts), d), np.float32)
    l2e = np.float32(math.log2(math.e))
    for o, t0 in enumerate(starts):
        X = gate[t0:t0 + P] * l2e
        V = key[t0:t0 + P]
        M = X.max(axis=0)
        E = np.exp2(X - M)
        Z = np.zeros(d, np.float32)
        for e in E:
            Z = Z + e
        R = np.float32(1.0) / Z
        acc = np.zeros(d, np.float32)
        for e, v in zip(E, V):
            if compress:
                pb = ts.bf16_bits_to_f32(ts.f32_to_bf16_bits(e * R))
                acc = acc + ts.bf16_bits_to_f32(ts.f32_to_bf16_bits(pb * v))
            else:
                acc = acc + e * v
        out[o] = acc if compress else acc * R
    return out


KPOOL_MASS_PACKS = {
    "p4_d64": lambda: ts.make_kpool_custom([64, 37, 12, 3, 29], pool=4, d=64, leads=[1, 0, 2, 0, 3],
                                           seed=31),
    "p2_d64_x4": lambda: ts.make_kpool_custom([40, 21], pool=2, d=64, seed=32, gate_scale=4.0),
    "p8_d32_x4": lambda: ts.make_kpool_custom([96, 41], pool=8, d=32, leads=[5, 0], seed=33,
                                              gate_scale=4.0),
    "p16_d16": lambda: ts.make_kpool_custom([160, 70], pool=16, d=16, seed=34),
    "p64_d8_x4": lambda: ts.make_kpool_custom([256, 200], pool=64, d=8, seed=35, gate_scale=4.0),
}


@pytest.mark.parametrize("name", sorted(KPOOL_MASS_PACKS))
@pytest.mark.parametrize("compress", [False, True])
def test_fp32_evaluation_within_mass_and_slack(oracle_lib, name, compress):
    """A plain float32 evaluation of every pool differs from the fp64 value by at most
    KAPPA * u32 * mass + slack (pools of 2 to 64 keys, sharpened gates included)."""
    pack = KPOOL_MASS_PACKS[name]()
    r = oracle.kpool_fwd_pack(pack, compress=compress, want_f64=True, want_err=True)
    got = f32_kpool(pack, compress).astype(np.float64)
    dev = np.abs(got - r["out_f64"]) - r["out_slack"]
    assert (dev <= KAPPA * U32 * r["out_err"]).all(), float(
        np.max(dev / (U32 * r["out_err"] + 1e-300)))
    if not compress:
        assert (r["out_slack"] == 0).all()


def test_slack_marks_undecided_weights(oracle_lib):
    slack_sweep(None)


def slack_sweep(lib):
    """Pools of two keys with gates (0, g) over every bf16 g in [-4, 4]: the weight of the
    second key is exactly sigma(g). Where sigma(g) lies within a narrow band around a bf16
    rounding boundary (a tie of two bf16 neighbours) the slack must be non-zero; well away
    from every boundary it must be zero."""
    gs = np.unique(ts.bf16_bits_to_f32(np.arange(0, 1 << 16, dtype=np.uint16)))
    gs = gs[np.isfinite(gs) & (np.abs(gs) <= 4)].astype(np.float64)
    n = gs.size
    cu = np.arange(0, 2 * n + 1, 2, dtype=np.int32)
    gate = np.zeros((2 * n, 1), np.float32)
    gate[1::2, 0] = gs
    key = np.ones((2 * n, 1), np.float32) * np.float32(1.5)
    pack = ts.KPoolPack("sweep", 2, 1, 2 * n, cu, None, ts.f32_to_bf16_bits(key),
                        ts.f32_to_bf16_bits(gate))
    r = oracle.kpool_fwd_pack(pack, compress=True, want_err=True, lib=lib)
    slack = r["out_slack"].reshape(-1)
    # distance of each weight to the nearest bf16 tie, relative to the weight
    near = np.zeros(n, bool)
    far = np.zeros(n, bool)
    for i, g in enumerate(gs):
        for p in (1.0 / (1.0 + math.exp(g)), 1.0 / (1.0 + math.exp(-g))):
            e = math.frexp(p)[1]
            step = 2.0 ** (e - 8)                       # bf16 spacing around p
            tie = (math.floor(p / step - 0.5) + 0.5) * step
            rel = min(abs(p - tie), abs(p - tie - step)) / p
            if rel < 1e-7:
                near[i] = True                           # inside any evaluation window
            if rel < 1e-4:
                far[i] = True                            # (not far)
    far = ~far
    assert near.any(), "no weight near a bf16 tie in the sweep"
    assert (slack[near] > 0).all()
    assert (slack[far] == 0).all()


# ----------------------------------------------------------------------------------
# All pins against one oracle library (the planted-mistake tests run them on mutants)
# ----------------------------------------------------------------------------------

def kpool_pin_failures(lib):
    """Names of the KPool pins that the oracle library ``lib`` fails."""
    failed = []
    for k, pack in enumerate(kpool_tiny_packs()):
        for compress in (False, True):
            bf, _ = brute_kpool(pack, compress)
            try:
                r = oracle.kpool_fwd_pack(pack, compress=compress, want_f64=True, lib=lib)
            except oracle.OracleError:
                failed.append(f"error{k}{compress}")
                continue
            if r["out"].shape != bf.shape or not np.allclose(r["out_f64"], bf, rtol=1e-13,
                                                              atol=1e-15):
                failed.append(f"brute{k}{compress}")
    with open(os.path.join(GOLDEN, "kpool_hand.json")) as fh:
        gd = json.load(fh)
    env = {"e": math.e, "__builtins__": {}}
    for ex in gd["examples"]:
        key = ts.f32_to_bf16_bits(np.array(ex["key"], np.float32))
        gate = ts.f32_to_bf16_bits(np.array(ex["gate"], np.float32))
        cu = np.array(ex["cu_seqlens"], np.int32)
        lead = None if ex["lead"] is None else np.array(ex["lead"], np.int32)
        for mode, want in ex["expected"].items():
            try:
                r = oracle.kpool_fwd(key, gate, cu, lead, ex["P"], ex["d"], int(cu[-1]),
                                     compress=mode == "compress", want_f64=True, want_err=True,
                                     lib=lib)
            except oracle.OracleError:
                failed.append(f"golden_error_{ex['name']}")
                continue
            vals = [float(Fraction(s)) if "e" not in s else eval(s, env) for s in want["out_f64"]]
            if r["out_f64"].size != len(vals) or not np.allclose(r["out_f64"].reshape(-1), vals,
                                                                 rtol=1e-15, atol=0):
                failed.append(f"golden_{ex['name']}_{mode}")
            if "out_err" in want and not np.allclose(
                    r["out_err"].reshape(-1), [eval(s, env) for s in want["out_err"]], rtol=1e-14):
                failed.append(f"golden_err_{ex['name']}")
    for name in ("p4_d64", "p8_d32_x4"):
        pack = KPOOL_MASS_PACKS[name]()
        for compress in (False, True):
            r = oracle.kpool_fwd_pack(pack, compress=compress, want_f64=True, want_err=True,
                                      lib=lib)
            got = f32_kpool(pack, compress).astype(np.float64)
            if got.shape != r["out_f64"].shape or not (
                    np.abs(got - r["out_f64"]) - r["out_slack"] <= KAPPA * U32 * r["out_err"]).all():
                failed.append(f"f32_{name}_{compress}")
    try:
        slack_sweep(lib)
    except AssertionError:
        failed.append("slack_sweep")
    return failed


def test_unmutated_oracle_passes_kpool_pins(oracle_lib):
    assert kpool_pin_failures(oracle.load()) == []
