"""Pins for the fp64 oracle, independent of the oracle's own code (CPU only).

Each test checks the oracle against something it cannot share a mistake with:

* a brute-force evaluator that finds each window's members by scanning every
  (token, column) slot of the pack against a membership predicate, instead of the
  oracle's index formulas;
* the closed form total_comp = sum floor(L_s / ratio), counted here by scanning
  tokens for block starts;
* invariants of the softmax pooling: equal scores give the window mean, a common
  shift of the scores changes nothing, the weights sum to one (sum of dKV over a
  window = dout), the softmax Jacobian rows sum to zero (sum of dScore over a
  window = 0, hence the dAPE columns of one output column sum to zero), and
  ratio=1 / coff=1 is the identity;
* central finite differences of L = sum(dout * out) in fp64;
* a hand-derived worked example (tests/golden/hand_pack_r2_c2.json);
* bf16 round-to-nearest-even against a brute-force nearest search over all bf16
  values.

The operation is the one described on "Megatron-LM PR #5984" (commits "CSA: add
fused Compressor forward+backward CuTe-DSL kernels", "fold dKV/dScore zero-init
into the backward kernel", "widen the validated envelope to coff in {1, 2}") and
"cudnn-frontend PR #710" (ratio=2 envelope).
"""
import bisect
import json
import math
import os

import numpy as np
import pytest

import oracle
import thd_synth as ts

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------------
# Independent brute-force evaluator (predicate formulation)
# ----------------------------------------------------------------------------------

def _bf(bits):
    return float(ts.bf16_bits_to_f32(np.array([bits], dtype=np.uint16))[0])


def brute_blocks(cu, r):
    """Complete blocks in token order, found by scanning: a token starts a block when
    its offset from its segment's start is a multiple of r and r tokens of the same
    segment follow from it (itself included)."""
    blocks = []
    S = len(cu) - 1
    for t in range(int(cu[0]), int(cu[S])):
        s = max(i for i in range(S) if cu[i] <= t < cu[i + 1]) if S else None
        if (t - cu[s]) % r == 0 and t + r <= cu[s + 1]:
            blocks.append((s, t))
    return blocks


def members(cu, r, coff, d, block, j, capacity):
    """Window members of output column j of ``block``, by testing every slot."""
    s, start = block
    C = coff * d
    own_col = d + j if coff == 2 else j
    has_prev = coff == 2 and start - r >= cu[s]
    out = []
    for t in range(capacity):
        for col in range(C):
            if start <= t < start + r and col == own_col:
                out.append((t, col, t - start))
            elif has_prev and start - r <= t < start and col == j:
                out.append((t, col, t - (start - r)))
    return out


def brute_force(pack):
    cu = [int(x) for x in pack.cu_seqlens]
    r, coff, d, cap = pack.ratio, pack.coff, pack.d, pack.capacity
    C = coff * d
    blocks = brute_blocks(cu, r)
    out = np.zeros((len(blocks), d))
    dkv = np.zeros((cap, C))
    dsc = np.zeros((cap, C))
    own = np.zeros((cap, C), dtype=np.int64)
    dape = np.zeros((r, C))
    for k, blk in enumerate(blocks):
        for j in range(d):
            mem = members(cu, r, coff, d, blk, j, cap)
            x = [_bf(pack.score[t, c]) + float(pack.ape[a, c]) for t, c, a in mem]
            v = [_bf(pack.kv[t, c]) for t, c, a in mem]
            m = max(x)
            e = [math.exp(xi - m) for xi in x]
            z = sum(e)
            p = [ei / z for ei in e]
            o = sum(pi * vi for pi, vi in zip(p, v))
            out[k, j] = o
            g = _bf(pack.dout[k, j]) if pack.dout.size else 0.0
            for (t, c, a), pi, vi in zip(mem, p, v):
                dkv[t, c] += pi * g
                dsc[t, c] += pi * g * (vi - o)
                own[t, c] += 1
                dape[a, c] += pi * g * (vi - o)
    return dict(out=out, dkv=dkv, dscore=dsc, owners=own, dape=dape, blocks=blocks)


def tiny_packs():
    return [
        ts.make_pack("tiny"),
        ts.make_custom([9, 0, 2, 7], ratio=2, coff=2, d=3, pad_rows=3, seed=1),
        ts.make_custom([5, 6], ratio=3, coff=1, d=2, pad_rows=2, seed=2),
        ts.make_custom([1, 8, 3], ratio=1, coff=2, d=2, pad_rows=1, seed=3),
        ts.make_custom([12, 4], ratio=4, coff=1, d=1, pad_rows=0, seed=4),
    ]


@pytest.fixture(scope="module", params=range(5), ids=["tiny", "r2c2", "r3c1", "r1c2", "r4c1"])
def pack_and_brute(request, oracle_lib):
    pack = tiny_packs()[request.param]
    return pack, brute_force(pack)


def test_total_comp_closed_form(oracle_lib):
    pack = ts.make_pack("tiny")
    assert oracle.total_comp(pack.cu_seqlens, 4) == 9 + 3 + 0 == 12
    rng = np.random.default_rng(11)
    for _ in range(40):
        S = int(rng.integers(0, 7))
        lens = rng.integers(0, 30, size=S)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        r = int(rng.integers(1, 9))
        assert oracle.total_comp(cu, r) == len(brute_blocks(list(cu), r))


def test_map_blocks_matches_scan(oracle_lib):
    rng = np.random.default_rng(12)
    for _ in range(30):
        S = int(rng.integers(1, 6))
        lens = rng.integers(0, 25, size=S)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        r = int(rng.integers(1, 6))
        blocks = brute_blocks(list(cu), r)
        m = oracle.map_blocks(cu, r, len(blocks) + 2)
        for o, (s, start) in enumerate(blocks):
            assert tuple(m[o]) == (s, (start - cu[s]) // r, start)
        assert (m[len(blocks):] == -1).all()


def test_forward_matches_brute_force(pack_and_brute):
    pack, bf = pack_and_brute
    f = oracle.fwd_pack(pack, want_f64=True)
    np.testing.assert_allclose(f["out_f64"], bf["out"], rtol=1e-13, atol=1e-15)
    assert (f["out"] == oracle.round_bf16(bf["out"])).all()


def test_backward_matches_brute_force(pack_and_brute):
    pack, bf = pack_and_brute
    b = oracle.bwd_pack(pack, want_f64=True, want_owners=True)
    assert (b["owners"] == bf["owners"]).all()
    np.testing.assert_allclose(b["dkv_f64"], bf["dkv"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(b["dscore_f64"], bf["dscore"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(b["dape_f64"], bf["dape"], rtol=1e-12, atol=1e-14)
    # unconsumed slots are exact +0 (bit pattern 0x0000), consumed ones carry the value
    zero = bf["owners"] == 0
    assert (b["dkv"][zero] == 0).all() and (b["dscore"][zero] == 0).all()
    assert (b["dkv"] == oracle.round_bf16(bf["dkv"])).all()
    assert (b["dape_f32"] == b["dape_f64"].astype(np.float32)).all()


def test_zero_classes_tiny(oracle_lib):
    """Tiny pack: segments 37, 12, 3 at ratio 4, coff 2, d 8, capacity 64. Count the
    unconsumed slots class by class, by hand."""
    pack = ts.make_pack("tiny")
    b = oracle.bwd_pack(pack, want_owners=True)
    own = b["owners"]
    d = 8
    # class (i): first-half columns of each segment's last block's own tokens
    last_blocks = [(32, 36), (45, 49)]      # seg 0: blocks 0..8 -> last = tokens 32..35
    for lo, hi in last_blocks:
        assert (own[lo:hi, :d] == 0).all() and (own[lo:hi, d:] == 1).all()
    # class (ii): tail token 36 of segment 0 (37 mod 4 = 1); segment 1 has no tail
    assert (own[36] == 0).all()
    # class (iii): segment 2 (3 tokens < ratio)
    assert (own[49:52] == 0).all()
    # class (iv): padding rows 52..63
    assert (own[52:] == 0).all()
    # consumed: seg 0 tokens 0..31 both halves, tokens 32..35 second half; seg 1 tokens
    # 37..44 both halves, 45..48 second half
    assert (own[0:32] == 1).all() and (own[37:45] == 1).all()
    assert int(own.sum()) == 8 * 4 * (2 * 9 - 1) + 8 * 4 * (2 * 3 - 1)


def test_uniform_scores_give_window_mean(oracle_lib):
    for coff in (1, 2):
        pack = ts.make_custom([11, 6], ratio=3, coff=coff, d=4, pad_rows=2, seed=5)
        pack.score[:] = ts.f32_to_bf16_bits(np.full(pack.score.shape, 0.75, np.float32))
        pack.ape[:] = 0.0
        f = oracle.fwd_pack(pack, want_f64=True)
        kv = ts.bf16_bits_to_f32(pack.kv).astype(np.float64)
        d, r = pack.d, pack.ratio
        o = 0
        for s in range(2):
            c = int(pack.cu_seqlens[s])
            n = (int(pack.cu_seqlens[s + 1]) - c) // r
            for b in range(n):
                own = kv[c + b * r:c + (b + 1) * r, (d if coff == 2 else 0):][:, :d]
                vals = [own]
                if coff == 2 and b >= 1:
                    vals.append(kv[c + (b - 1) * r:c + b * r, :d])
                mean = np.concatenate(vals, axis=0).mean(axis=0)
                np.testing.assert_allclose(f["out_f64"][o], mean, rtol=1e-14, atol=1e-15)
                o += 1


def test_common_score_shift_changes_nothing(oracle_lib):
    pack = ts.make_custom([10, 7], ratio=2, coff=2, d=3, seed=6)
    pack.ape[:] = np.round(pack.ape * 1024) / 1024  # shift by 0.25 stays exact in fp32
    f0 = oracle.fwd_pack(pack, want_f64=True)
    b0 = oracle.bwd_pack(pack, want_f64=True)
    pack.ape[:] += np.float32(0.25)
    f1 = oracle.fwd_pack(pack, want_f64=True)
    b1 = oracle.bwd_pack(pack, want_f64=True)
    np.testing.assert_allclose(f1["out_f64"], f0["out_f64"], rtol=1e-15, atol=1e-16)
    np.testing.assert_allclose(b1["dscore_f64"], b0["dscore_f64"], rtol=1e-14, atol=1e-16)


def test_softmax_identities(oracle_lib):
    """Per window: sum of dKV = dout (weights sum to one); sum of dScore = 0."""
    pack = ts.make_custom([13, 9, 2], ratio=4, coff=2, d=5, pad_rows=4, seed=7)
    b = oracle.bwd_pack(pack, want_f64=True)
    m = oracle.map_blocks(pack.cu_seqlens, pack.ratio, pack.total_comp)
    r, d = pack.ratio, pack.d
    g = ts.bf16_bits_to_f32(pack.dout).astype(np.float64)
    for o, (s, blk, base) in enumerate(m):
        for j in range(d):
            slots = [(base + w, d + j) for w in range(r)]
            if blk >= 1:
                slots += [(base - r + w, j) for w in range(r)]
            sk = sum(b["dkv_f64"][t, c] for t, c in slots)
            ss = sum(b["dscore_f64"][t, c] for t, c in slots)
            mag = sum(abs(b["dscore_f64"][t, c]) for t, c in slots)
            assert abs(sk - g[o, j]) <= 1e-14 * max(1.0, abs(g[o, j]))
            assert abs(ss) <= 1e-14 * max(mag, 1e-300)
    # hence each output column's dAPE entries (both halves) sum to zero
    col = b["dape_f64"][:, :d].sum(axis=0) + b["dape_f64"][:, d:].sum(axis=0)
    assert np.all(np.abs(col) <= 1e-13 * np.abs(b["dape_f64"]).sum())


def test_ratio_one_is_identity(oracle_lib):
    pack = ts.make_custom([5, 3], ratio=1, coff=1, d=6, pad_rows=2, seed=8)
    f = oracle.fwd_pack(pack)
    b = oracle.bwd_pack(pack, want_f64=True)
    T = int(pack.cu_seqlens[-1])
    assert (f["out"] == pack.kv[:T]).all()
    assert (b["dkv"][:T] == pack.dout).all()
    assert (b["dscore_f64"] == 0).all() and (b["dape_f64"] == 0).all()
    assert (b["dkv"][T:] == 0).all()


@pytest.mark.parametrize("coff", [1, 2])
def test_finite_differences(oracle_lib, coff):
    """Central differences of L = sum(dout * out_unrounded) with a power-of-two step
    around elements set to zero (so that +-h is exact in bf16 and fp32)."""
    pack = ts.make_custom([9, 6], ratio=3, coff=coff, d=2, pad_rows=1, seed=9)
    g = ts.bf16_bits_to_f32(pack.dout).astype(np.float64)
    h = 2.0 ** -14
    rng = np.random.default_rng(3)

    def loss(p):
        return float((oracle.fwd_pack(p, want_f64=True)["out_f64"] * g).sum())

    T = int(pack.cu_seqlens[-1])
    C = pack.C
    checks = 0
    for _ in range(12):
        t, c = int(rng.integers(0, T)), int(rng.integers(0, C))
        for name in ("kv", "score"):
            arr = getattr(pack, name)
            arr[t, c] = 0
            b = oracle.bwd_pack(pack, want_f64=True)
            grad = b["dkv_f64" if name == "kv" else "dscore_f64"][t, c]
            arr[t, c] = ts.f32_to_bf16_bits(np.array([h], np.float32))[0]
            lp = loss(pack)
            arr[t, c] = ts.f32_to_bf16_bits(np.array([-h], np.float32))[0]
            lm = loss(pack)
            arr[t, c] = 0
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad) <= 1e-7 * max(1.0, abs(grad)), (name, t, c, fd, grad)
            checks += 1
    for k in range(pack.ratio):
        for c in range(C):
            pack.ape[k, c] = 0.0
            b = oracle.bwd_pack(pack, want_f64=True)
            grad = b["dape_f64"][k, c]
            pack.ape[k, c] = h
            lp = loss(pack)
            pack.ape[k, c] = -h
            lm = loss(pack)
            pack.ape[k, c] = 0.0
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad) <= 1e-7 * max(1.0, abs(grad)), ("ape", k, c, fd, grad)
            checks += 1
    assert checks > 20


def test_golden_hand_pack(oracle_lib):
    with open(os.path.join(GOLDEN, "hand_pack_r2_c2.json")) as fh:
        gd = json.load(fh)
    env = {"e": math.e, "__builtins__": {}}
    ev = lambda s: eval(s, env)  # closed forms in e only
    cap, C = gd["capacity"], gd["coff"] * gd["d"]
    kv = ts.f32_to_bf16_bits(np.array(gd["kv"], np.float32))
    score = ts.f32_to_bf16_bits(np.array(gd["score"], np.float32))
    ape = np.array(gd["ape"], np.float32)
    dout = ts.f32_to_bf16_bits(np.array(gd["dout"], np.float32))
    cu = np.array(gd["cu_seqlens"], np.int32)
    r, coff, d = gd["ratio"], gd["coff"], gd["d"]
    f = oracle.fwd(kv, score, ape, cu, r, coff, d, cap, want_f64=True)
    b = oracle.bwd(kv, score, ape, cu, dout, r, coff, d, cap, want_f64=True, want_owners=True)
    exp = gd["expected"]
    np.testing.assert_allclose(f["out_f64"][:, 0], [ev(s) for s in exp["out"]], rtol=1e-15)
    assert [int(x) for x in f["out"][:, 0]] == [int(s, 16) for s in exp["out_bits"]]
    want_dkv = np.array([[ev(s) for s in row] for row in exp["dkv"]])
    want_dsc = np.array([[ev(s) for s in row] for row in exp["dscore"]])
    want_dape = np.array([[ev(s) for s in row] for row in exp["dape"]])
    np.testing.assert_allclose(b["dkv_f64"], want_dkv, rtol=1e-15, atol=0)
    np.testing.assert_allclose(b["dscore_f64"], want_dsc, rtol=1e-14, atol=0)
    np.testing.assert_allclose(b["dape_f64"], want_dape, rtol=1e-14, atol=0)
    assert (b["dkv"][want_dkv == 0] == 0).all() and (b["dscore"][want_dsc == 0] == 0).all()
    assert cap * C == 14 and int(b["owners"].sum()) == 6


# ----------------------------------------------------------------------------------
# The error masses (the parity tolerance's first-order fp32 error sizes)
# ----------------------------------------------------------------------------------

U32 = 2.0 ** -24


def golden_mass_mismatches(lib=None):
    """Names of the error masses of the hand-derived golden pack that the oracle (`lib`)
    gets wrong: out_err, dkv_err, dscore_err, dape_err against closed forms in e worked
    out by hand (tests/golden/hand_pack_r2_c2.json)."""
    with open(os.path.join(GOLDEN, "hand_pack_r2_c2.json")) as fh:
        gd = json.load(fh)
    env = {"e": math.e, "__builtins__": {}}
    for k, v in gd["definitions"].items():
        env[k] = eval(v, env)
    kv = ts.f32_to_bf16_bits(np.array(gd["kv"], np.float32))
    score = ts.f32_to_bf16_bits(np.array(gd["score"], np.float32))
    ape = np.array(gd["ape"], np.float32)
    dout = ts.f32_to_bf16_bits(np.array(gd["dout"], np.float32))
    cu = np.array(gd["cu_seqlens"], np.int32)
    r, coff, d, cap = gd["ratio"], gd["coff"], gd["d"], gd["capacity"]
    try:
        f = oracle.fwd(kv, score, ape, cu, r, coff, d, cap, want_err=True, lib=lib)
        b = oracle.bwd(kv, score, ape, cu, dout, r, coff, d, cap, want_err=True, lib=lib)
    except oracle.OracleError as ex:
        return [f"error: {ex}"]
    em = gd["expected_error_masses"]
    bad = []
    if not np.allclose(f["out_err"][:, 0], [eval(x, env) for x in em["out_err"]], rtol=1e-14,
                       atol=0):
        bad.append("out_err")
    for key in ("dkv_err", "dscore_err", "dape_err"):
        want = np.array([[eval(x, env) for x in row] for row in em[key]])
        if not np.allclose(b[key], want, rtol=1e-14, atol=0):
            bad.append(key)
    return bad


def test_error_masses_golden(oracle_lib):
    assert golden_mass_mismatches() == []


def f32_evaluation(pack):
    """Every window evaluated in plain float32 (numpy, one rounding per operation, the
    sums in window order), with window membership from brute_blocks (block starts found
    by scanning), not from the oracle. Also the fp64 weights' |p|-weighted |kv| sums."""
    cu = [int(x) for x in pack.cu_seqlens]
    r, coff, d, C = pack.ratio, pack.coff, pack.d, pack.C
    kv = ts.bf16_bits_to_f32(pack.kv)
    sc = ts.bf16_bits_to_f32(pack.score)
    ape = pack.ape.astype(np.float32)
    g = ts.bf16_bits_to_f32(pack.dout)
    blocks = brute_blocks(cu, r)
    out = np.zeros((len(blocks), d), np.float32)
    dkv = np.zeros((pack.capacity, C), np.float32)
    dsc = np.zeros((pack.capacity, C), np.float32)
    terms = np.zeros((len(blocks), r, C), np.float32)  # dScore terms per block and ape entry
    abs_mean = np.zeros((len(blocks), d))               # sum_w p_w |kv_w| in fp64
    for o, (s, start) in enumerate(blocks):
        pos = []
        if coff == 2 and start - r >= cu[s]:
            pos += [(start - r + w, 0, w) for w in range(r)]
        pos += [(start + w, d if coff == 2 else 0, w) for w in range(r)]
        X = np.stack([sc[t, c:c + d] + ape[w, c:c + d] for t, c, w in pos])
        V = np.stack([kv[t, c:c + d] for t, c, w in pos])
        M = X.max(axis=0)
        E = np.exp(X - M)
        Z = np.zeros(d, np.float32)
        for e in E:
            Z = Z + e
        P = E / Z
        O = np.zeros(d, np.float32)
        for p_, v in zip(P, V):
            O = O + p_ * v
        out[o] = O
        for (t, c, w), p_, v in zip(pos, P, V):
            k = p_ * g[o]
            dkv[t, c:c + d] = k
            dsc[t, c:c + d] = k * (v - O)
            terms[o, w, c:c + d] = dsc[t, c:c + d]
        X64 = X.astype(np.float64)
        P64 = np.exp(X64 - X64.max(axis=0))
        P64 /= P64.sum(axis=0)
        abs_mean[o] = (P64 * np.abs(V.astype(np.float64))).sum(axis=0)
    dape = terms.sum(axis=0, dtype=np.float32)  # numpy's pairwise float32 sum over blocks
    return dict(out=out, dkv=dkv, dscore=dsc, dape=dape, abs_mean=abs_mean)


MASS_PACKS = {
    "r4c2_d64": lambda: ts.make_custom([37, 12, 3, 29, 40], ratio=4, coff=2, d=64, pad_rows=3,
                                       seed=1),
    "r2c2_d64": lambda: ts.make_custom([20, 9, 31, 1], ratio=2, coff=2, d=64, seed=3),
    "r16c1_x4": lambda: ts.make_custom([64, 50, 33], ratio=16, coff=1, d=64, pad_rows=2, seed=2,
                                       score_scale=4.0),
    "r64c2_x4": lambda: ts.make_custom([300, 130], ratio=64, coff=2, d=32, seed=4,
                                       score_scale=4.0),
    "r128c1_x4": lambda: ts.make_custom([512, 300], ratio=128, coff=1, d=16, seed=5,
                                        score_scale=4.0),
    "r128c2_x4": lambda: ts.make_custom([600, 256], ratio=128, coff=2, d=8, seed=6,
                                        score_scale=4.0),
}
KAPPA_F32 = 8.0  # a plain float32 evaluation stays within KAPPA_F32 * u32 * mass


@pytest.mark.parametrize("name", sorted(MASS_PACKS))
def test_fp32_evaluation_within_error_masses(oracle_lib, name):
    """The masses are large enough: a plain float32 evaluation of every window (windows of
    4 to 256 positions, sharpened scores included) differs from the fp64 result by at most
    KAPPA_F32 * u32 * mass, element by element, for out, dKV, dScore and dAPE. (A mass that
    drops a term, e.g. the exponent-argument factor, fails here on the long windows.)"""
    pack = MASS_PACKS[name]()
    f = oracle.fwd_pack(pack, want_f64=True, want_err=True)
    b = oracle.bwd_pack(pack, want_f64=True, want_err=True, want_owners=True)
    e = f32_evaluation(pack)
    own = b["owners"] > 0
    checks = [("out", e["out"], f["out_f64"], f["out_err"]),
              ("dkv", e["dkv"][own], b["dkv_f64"][own], b["dkv_err"][own]),
              ("dscore", e["dscore"][own], b["dscore_f64"][own], b["dscore_err"][own]),
              ("dape", e["dape"], b["dape_f64"], b["dape_err"])]
    for label, got, ref, mass in checks:
        ratio = np.abs(got.astype(np.float64) - ref) / (U32 * mass + 1e-300)
        assert ratio.max() <= KAPPA_F32, (label, float(ratio.max()))


def test_error_masses_cover_summand_magnitudes(oracle_lib):
    """The masses are at least the magnitudes an fp32 evaluation rounds: out_err >= the
    weighted absolute kv sum sum_w p_w |kv_w| (so it is never below one rounding of each
    summand); dkv_err >= |dKV|; dscore_err >= |p g| sum_w p_w |kv_w| (the output's error
    enters through kv - out); dape_err >= the sum of |terms|; all are exactly 0 on
    unconsumed slots."""
    for name in ("r4c2_d64", "r16c1_x4"):
        pack = MASS_PACKS[name]()
        f = oracle.fwd_pack(pack, want_f64=True, want_err=True)
        b = oracle.bwd_pack(pack, want_f64=True, want_err=True, want_owners=True)
        e = f32_evaluation(pack)
        assert (f["out_err"] >= e["abs_mean"] * (1 - 1e-12)).all()
        own = b["owners"] > 0
        assert (b["dkv_err"][own] >= np.abs(b["dkv_f64"][own])).all()
        assert (b["dkv_err"][~own] == 0).all() and (b["dscore_err"][~own] == 0).all()
        assert (b["dape_err"] >= b["dape_abs"]).all()
        # dScore: every consumed slot's mass covers |p g| times its row's sum_w p_w |kv_w|
        m = oracle.map_blocks(pack.cu_seqlens, pack.ratio, pack.total_comp)
        g = ts.bf16_bits_to_f32(pack.dout).astype(np.float64)
        r, d = pack.ratio, pack.d
        for o, (s, blk, base) in enumerate(m[:8]):
            cols = slice(d, 2 * d) if pack.coff == 2 else slice(0, d)
            for w in range(r):
                pg = np.abs(b["dkv_f64"][base + w, cols])
                assert (b["dscore_err"][base + w, cols] >= pg * e["abs_mean"][o] * (1 - 1e-12)).all()


# ----------------------------------------------------------------------------------
# bf16 rounding against a brute-force nearest search
# ----------------------------------------------------------------------------------

def _all_positive_bf16():
    bits = np.arange(0x0000, 0x7F80, dtype=np.uint16)   # +0 .. largest finite
    vals = ts.bf16_bits_to_f32(bits).astype(np.float64)
    return list(vals) + [2.0 ** 128], list(range(0x0000, 0x7F80)) + [0x7F80]


def _nearest_bf16(x, vals, bits):
    if x == 0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    i = bisect.bisect_left(vals, a)
    if i < len(vals) and vals[i] == a:
        k = i
    else:
        lo, hi = i - 1, min(i, len(vals) - 1)
        if a >= vals[-1]:
            k = len(vals) - 1
        elif a - vals[lo] < vals[hi] - a:
            k = lo
        elif a - vals[lo] > vals[hi] - a:
            k = hi
        else:
            k = lo if bits[lo] % 2 == 0 else hi
    return bits[k] | (0x8000 if x < 0 else 0)


def test_bf16_rounding_brute_force(oracle_lib):
    vals, bits = _all_positive_bf16()
    rng = np.random.default_rng(5)
    xs = list(rng.standard_normal(3000) * np.exp2(rng.integers(-140, 130, 3000)))
    # exact ties between neighbours (even and odd), subnormals, overflow boundary
    for k in rng.integers(1, 0x7F7F, 400):
        xs.append((vals[k] + vals[k + 1]) / 2)
        xs.append(-(vals[k] + vals[k + 1]) / 2)
    xs += [2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 2.0 ** -126 * 0.75, 1e-45,
           vals[0x7F7F], (vals[0x7F7F] + 2.0 ** 128) / 2, 2.0 ** 128 * 0.999, 1.0, -0.0]
    xs = np.array(xs, dtype=np.float64)
    got = oracle.round_bf16(xs)
    want = np.array([_nearest_bf16(float(x), vals, bits) for x in xs], dtype=np.uint16)
    assert (got == want).all(), xs[got != want][:5]


def test_oracle_rejects_bad_inputs(oracle_lib):
    pack = ts.make_pack("tiny")
    bad = pack.cu_seqlens.copy()
    bad[2] = bad[1] - 1
    with pytest.raises(oracle.OracleError):
        oracle.fwd(pack.kv, pack.score, pack.ape, bad, 4, 2, 8, pack.capacity)
    big = pack.cu_seqlens.copy()
    big[-1] = pack.capacity + 1
    with pytest.raises(oracle.OracleError):
        oracle.bwd(pack.kv, pack.score, pack.ape, big, pack.dout, 4, 2, 8, pack.capacity)
    with pytest.raises(oracle.OracleError):
        oracle.fwd(pack.kv, pack.score, pack.ape, pack.cu_seqlens, 4, 2, 8, pack.capacity,
                   out_rows=11)


def test_threaded_oracle_matches_single_thread(oracle_lib):
    """The multi-threaded drivers (used to time the oracle on every host core) give the
    single-thread results: out, dKV, dScore bit for bit, dAPE up to the order of the final
    additions of the per-thread sums."""
    packs = [ts.make_custom([37, 12, 3, 0, 29], ratio=4, coff=2, d=8, pad_rows=5, seed=21),
             ts.make_custom([9, 40, 1, 17], ratio=3, coff=1, d=5, pad_rows=2, seed=22)]
    for pack in packs:
        f1 = oracle.fwd_pack(pack)["out"]
        b1 = oracle.bwd_pack(pack)
        for nt in (1, 2, 3, 7):
            assert (oracle.fwd_threads(pack, nt) == f1).all()
            bt = oracle.bwd_threads(pack, nt)
            assert (bt["dkv"] == b1["dkv"]).all() and (bt["dscore"] == b1["dscore"]).all()
            np.testing.assert_allclose(bt["dape_f64"], b1["dape_f64"], rtol=1e-13, atol=1e-16)
    assert oracle.hardware_threads() >= 1
