"""Bounded waits, exercised without any fault.

Every pipeline wait of the bulk-copy kernels (block streaming, long window) gives up after
a bound, records CSA_DEVERR_TIMEOUT in the device error word, lets the copies its CTA has
issued land, and returns. The test hook csa_compressor_test_hooks shortens the bound to
about 10 ms and makes the producer of the first CTA skip the copies of one row, so that
the waits for that stage run out (a stage that nothing fills). Checked, through the C ABI:

* the call returns and the error word reads CSA_DEVERR_TIMEOUT;
* the slots only the withheld row writes keep their NaN prefill, and every other output
  is bit for bit what a normal call writes;
* the next call on the same stream (hooks off) matches the fp64 oracle.
"""
import numpy as np
import pytest

import oracle
import thd_synth as ts
from tests import gpu_harness as H
from tests.parity import compare_bf16

pytestmark = pytest.mark.gpu

WAIT_CYCLES = 20_000_000  # about 10 ms at GB300 clocks

# name -> (pack, direction); each shape takes a bulk-copy kernel, and the first CTA's
# range starts with row 0 (segment 0, block 0), which is the row withheld
CASES = {
    "stream_bwd": (lambda: ts.make_pack("tiny"), "bwd"),
    "stream_fwd": (lambda: ts.make_custom([12, 8], ratio=4, coff=2, d=512, pad_rows=2, seed=60),
                   "fwd"),
    # (long windows: one 32-column slice, so that row 0 lies in the first CTA alone)
    "long_bwd": (lambda: ts.make_custom([50, 16, 5], ratio=16, coff=1, d=32, pad_rows=3, seed=61),
                 "bwd"),
    "long_fwd": (lambda: ts.make_custom([50, 16, 5], ratio=16, coff=1, d=32, pad_rows=3, seed=61),
                 "fwd"),
    # 256-position windows
    "long256_bwd": (lambda: ts.make_custom([300, 128], ratio=128, coff=2, d=32, pad_rows=1,
                                           seed=62), "bwd"),
    "long256_fwd": (lambda: ts.make_custom([300, 128], ratio=128, coff=2, d=32, pad_rows=1,
                                           seed=62), "fwd"),
}


def _row0_slots(pack):
    """(token, column) slots that row 0 (segment 0's first block) alone writes: its own
    block's tokens at its own-half columns (a first block has no previous half)."""
    mask = np.zeros((pack.capacity, pack.C), dtype=bool)
    c0 = int(pack.cu_seqlens[0])
    lo = pack.d if pack.coff == 2 else 0
    mask[c0:c0 + pack.ratio, lo:lo + pack.d] = True
    return mask


def _run(gp, pack, direction, dev):
    if direction == "fwd":
        out, err = H.run_fwd(gp, pack, dev=dev, prefill_bits=H.BF16_NAN)
        return (out,), err
    dkv, dsc, _, err = H.run_bwd(gp, pack, dev=dev, prefill_bits=H.BF16_NAN)
    return (dkv, dsc), err


@pytest.mark.parametrize("name", sorted(CASES))
def test_wait_runs_out_and_kernel_returns(cuda_lib, name):
    make, direction = CASES[name]
    pack = make()
    dev = H.device_pack(pack)
    normal, err = _run(cuda_lib, pack, direction, dev)
    assert err == 0
    cuda_lib.csa_compressor_test_hooks(WAIT_CYCLES, 0)
    try:
        stopped, err = _run(cuda_lib, pack, direction, dev)
    finally:
        cuda_lib.csa_compressor_test_hooks(0, -1)
    assert err == cuda_lib.CSA_DEVERR_TIMEOUT
    if direction == "fwd":
        got = stopped[0].reshape(pack.total_comp, pack.d)
        want = normal[0].reshape(pack.total_comp, pack.d)
        assert (got[0] == H.BF16_NAN).all()  # the withheld row was never written
        assert (got[1:] == want[1:]).all()
    else:
        skip = _row0_slots(pack)
        for got, want in zip(stopped, normal):
            got = got.reshape(pack.capacity, pack.C)
            want = want.reshape(pack.capacity, pack.C)
            assert (got[skip] == H.BF16_NAN).all()
            assert (got[~skip] == want[~skip]).all()
    # the next call on the same stream runs normally and matches the oracle
    again, err = _run(cuda_lib, pack, direction, dev)
    assert err == 0
    if direction == "fwd":
        ref = oracle.fwd_pack(pack, want_f64=True, want_err=True)
        rep = compare_bf16("out", again[0], ref["out"], ref["out_f64"], ref["out_err"])
        assert rep.fail == 0, str(rep)
    else:
        ref = oracle.bwd_pack(pack, want_f64=True, want_err=True)
        for label, got, key, err_mass in (("dkv", again[0], "dkv", ref["dkv_err"]),
                                          ("dscore", again[1], "dscore", ref["dscore_err"])):
            rep = compare_bf16(label, got, ref[key], ref[key + "_f64"], err_mass)
            assert rep.fail == 0, str(rep)
