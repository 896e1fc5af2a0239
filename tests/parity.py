"""Element-wise comparison of CUDA results with the oracle, with the tolerance the
arithmetic allows.

out, dKV, dScore (bf16): an element passes if
  (1) |gpu - bf16(ref)| <= ulp(bf16(ref))              -- one bf16 step of the fp64
      result rounded to bf16, or
  (2) |gpu - ref| <= ulp(ref) + KAPPA * u32 * err       -- for elements whose value
      cancels: err is the oracle's first-order error mass of an fp32 evaluation (the
      summands' magnitudes and the spread of kv around the output weighted by the
      exponent arguments, see oracle/csa_oracle.cpp), u32 = 2^-24.
dAPE (fp32): |gpu - ref| <= 1e-5 |ref| + KAPPA * u32 * err_dape.
ulp(y) is the bf16 spacing at |y| (2^(e-8) for |y| in [2^(e-1), 2^e)), and the
subnormal spacing 2^-133 at zero. KAPPA = 8: a plain float32 evaluation of every window
stays within 8 u32 x mass (pinned on the CPU for windows of 4..256 positions), and the
CUDA kernels used at most 5.3 on every parity pack (the per-pack record is kept with the
profiles). The report counts how many elements needed clause (2) and the largest kappa
one of them used; the tests cap the count.
"""
import dataclasses

import numpy as np

import thd_synth as ts

U32 = 2.0 ** -24
KAPPA = 8.0


def bits_to_f64(bits):
    return ts.bf16_bits_to_f32(bits).astype(np.float64)


def ulp_bf16(x):
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(ax)
    q = np.maximum(e - 8, -133).astype(np.float64)
    return np.where(ax > 0, np.exp2(q), 2.0 ** -133)


@dataclasses.dataclass
class Report:
    name: str
    n: int
    exact: int
    clause2: int
    fail: int
    worst: list
    kappa_used: float = 0.0  # largest kappa an element needing clause 2 required

    def __str__(self):
        return (f"{self.name}: n={self.n} bit-exact={self.exact} needed-clause2={self.clause2} "
                f"kappa-used={self.kappa_used:.2f} fail={self.fail} worst={self.worst[:3]}")


def compare_bf16(name, gpu_bits, ref_bits, ref_f64=None, err=None, kappa=KAPPA, slack=None):
    """Clause 1, else clause 2 (with `slack`, an absolute allowance the oracle gives where
    an intermediate rounding decision is not fixed by the arithmetic: KPool's compressed
    weights)."""
    gpu_bits = np.asarray(gpu_bits).reshape(-1)
    ref_bits = np.asarray(ref_bits).reshape(-1)
    g = bits_to_f64(gpu_bits)
    rb = bits_to_f64(ref_bits)
    exact = gpu_bits == ref_bits
    ok1 = np.abs(g - rb) <= ulp_bf16(rb)
    ok1 &= ~np.isnan(g)
    ok = ok1.copy()
    need2 = np.zeros_like(ok)
    kappa_used = 0.0
    if ref_f64 is not None and err is not None:
        ref = np.asarray(ref_f64).reshape(-1)
        e = np.asarray(err).reshape(-1)
        bad = ~ok1
        if bad.any():
            dev = np.abs(g[bad] - ref[bad]) - ulp_bf16(ref[bad])
            if slack is not None:
                dev = dev - np.asarray(slack).reshape(-1)[bad]
            tol = kappa * U32 * e[bad]
            ok2 = dev <= tol
            ok[bad] = ok2
            need2[np.flatnonzero(bad)[ok2]] = True
            if ok2.any():
                kappa_used = float(np.max(np.maximum(dev[ok2], 0) / (U32 * e[bad][ok2] + 1e-300)))
    idx = np.flatnonzero(~ok)
    worst = [(int(i), float(g[i]), float(rb[i])) for i in idx[:5]]
    return Report(name, int(g.size), int(exact.sum()), int(need2.sum()), int(idx.size), worst,
                  kappa_used)


def compare_dape(gpu, ref_f64, err, kappa=KAPPA, rel=1e-5):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref_f64).reshape(-1)
    e = np.asarray(err).reshape(-1)
    dev = np.abs(gpu - ref) - rel * np.abs(ref)
    tol = kappa * U32 * e
    ok = dev <= tol
    rel_ok = dev <= 0
    idx = np.flatnonzero(~ok)
    worst = [(int(i), float(gpu[i]), float(ref[i])) for i in idx[:5]]
    used = ok & ~rel_ok
    kappa_used = float(np.max(dev[used] / (U32 * e[used] + 1e-300))) if used.any() else 0.0
    return Report("dape", int(gpu.size), int(rel_ok.sum()), int(used.sum()), int(idx.size), worst,
                  kappa_used)
