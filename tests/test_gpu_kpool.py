"""KPool (the DSA indexer's key pooling) through the C ABI against the fp64 oracle.

The operation is the one on "Megatron-LM PR #8835" (the KPool commits): an FP32 softmax
of a gate over pools of P consecutive keys, the grid restarting at each segment's first
valid key, default FP32 weighted sum or key-dtype compression. Every output element is
compared with the oracle (tests/parity.py: one bf16 ulp, else the error mass plus, under
compression, the oracle's slack for weights whose bf16 rounding the arithmetic does not
fix). Packs cover the vector kernel (d % 8 == 0, P <= 8, aligned) and the scalar kernel
(other P, odd d, pointers off their 16-byte boundary), leads past a segment's end, empty
and short segments, padding rows, sharpened gates, the full-size packs of the bench, and
the device-side rejections.
"""
import numpy as np
import pytest

import oracle
import thd_synth as ts
from tests import gpu_harness as H
from tests.parity import compare_bf16
from tests.test_gpu_parity import log_reports

pytestmark = pytest.mark.gpu

CLAUSE2_CAP = 1e-4  # fraction of the elements allowed to need clause 2 (at least 2)


def run_kpool(gp, pack, compress, out_rows=None, shift=0, prefill=H.BF16_NAN, lead=None,
              cu=None):
    import torch
    dev = ts.kpool_to_torch(pack, "cuda")
    key, gate = dev["key"], dev["gate"]
    if shift:
        key, gate = H.shifted_copy(key, shift), H.shifted_copy(gate, shift)
    lead_t = dev.get("lead") if lead is None else torch.from_numpy(lead).cuda()
    cu_t = dev["cu_seqlens"] if cu is None else torch.from_numpy(cu).cuda()
    rows = pack.total_pools if out_rows is None else out_rows
    out = H.shifted_empty((max(rows, 1), pack.d), torch.int16, shift)
    out.fill_(np.int16(np.uint16(prefill).view(np.int16)))
    out = out.view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gp.csa_kpool_fwd(key, gate, cu_t, lead_t, pack.S, pack.pool, pack.d, pack.capacity, out,
                     rows, int(compress), err)
    torch.cuda.synchronize()
    return ts.bf16_tensor_bits(out)[:max(rows, 1)], int(err.item())


def check(gp, pack, compress, shift=0, label=None, nthreads=16):
    got, err = run_kpool(gp, pack, compress, shift=shift)
    assert err == 0
    n = pack.total_pools
    ref = oracle.kpool_fwd_pack(pack, compress=compress, want_f64=True, want_err=True,
                                nthreads=nthreads)
    rep = compare_bf16("out", got[:n], ref["out"], ref["out_f64"], ref["out_err"],
                       slack=ref["out_slack"])
    log_reports(label or f"{pack.name}{'+compress' if compress else ''}", rep)
    assert rep.fail == 0, str(rep)
    assert rep.clause2 <= max(2, CLAUSE2_CAP * rep.n), str(rep)
    return got


SMALL = {
    "tiny": lambda: ts.make_kpool("kpool_tiny"),
    "p1_d64": lambda: ts.make_kpool_custom([9, 0, 5], pool=1, d=64, leads=[2, 0, 5], seed=41),
    "p2_d128_x4": lambda: ts.make_kpool_custom([37, 12, 3, 1], pool=2, d=128, pad_rows=5,
                                               seed=42, gate_scale=4.0),
    "p3_d64": lambda: ts.make_kpool_custom([40, 7, 2, 31], pool=3, d=64, leads=[1, 0, 9, 4],
                                           seed=43),
    "p4_d136": lambda: ts.make_kpool_custom([64, 13, 22], pool=4, d=136, leads=[3, 1, 0],
                                            pad_rows=7, seed=44),
    "p5_d16": lambda: ts.make_kpool_custom([60, 26, 4, 11], pool=5, d=16, seed=45),
    "p8_d128_x4": lambda: ts.make_kpool_custom([200, 57, 8, 15], pool=8, d=128, leads=[7, 0, 0, 1],
                                               seed=46, gate_scale=4.0),
    "p8_d2048": lambda: ts.make_kpool_custom([48, 17], pool=8, d=2048, seed=47),
    # scalar kernel: pools above 8, odd head dims
    "p16_d64": lambda: ts.make_kpool_custom([100, 33, 16], pool=16, d=64, leads=[2, 0, 0],
                                            seed=48),
    "p64_d32_x4": lambda: ts.make_kpool_custom([300, 129], pool=64, d=32, seed=49, gate_scale=4.0),
    "p4_d65": lambda: ts.make_kpool_custom([30, 11, 9], pool=4, d=65, leads=[0, 3, 1], seed=50),
    "p3_d13": lambda: ts.make_kpool_custom([25, 8], pool=3, d=13, seed=51),
    "p4_d4096": lambda: ts.make_kpool_custom([16, 9], pool=4, d=4096, seed=52),
    # many short segments with leads
    "many_p4_d64": lambda: ts.make_kpool_custom(list(np.arange(2000) % 13), pool=4, d=64,
                                                leads=list(np.arange(2000) % 5), pad_rows=9,
                                                seed=53),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("compress", [False, True])
def test_kpool_small(cuda_lib, name, compress):
    check(cuda_lib, SMALL[name](), compress, label=f"kpool_{name}{'+compress' if compress else ''}")


@pytest.mark.parametrize("name", ["tiny", "p4_d136", "p8_d128_x4"])
@pytest.mark.parametrize("compress", [False, True])
def test_kpool_misaligned(cuda_lib, name, compress):
    """Tensors one element past a 16-byte boundary take the scalar kernel."""
    check(cuda_lib, SMALL[name](), compress, shift=1,
          label=f"kpool_{name}+misaligned{'+compress' if compress else ''}")


@pytest.mark.parametrize("name", ["kpool_16x8192_d128_p4", "kpool_ragged_d128_p4",
                                  "kpool_64x8192_d128_p4"])
@pytest.mark.parametrize("compress", [False, True])
def test_kpool_full(cuda_lib, name, compress):
    check(cuda_lib, ts.make_kpool(name), compress)


def test_kpool_rows_past_pools_untouched_and_repeatable(cuda_lib):
    pack = ts.make_kpool("kpool_ragged_d128_p4")
    a, err = run_kpool(cuda_lib, pack, False, out_rows=pack.total_pools + 5)
    assert err == 0
    assert (a[pack.total_pools:] == H.BF16_NAN).all()
    b, _ = run_kpool(cuda_lib, pack, False, out_rows=pack.total_pools + 5)
    assert (a == b).all()


@pytest.mark.parametrize("shift", [0, 1])
def test_kpool_device_rejections(cuda_lib, shift):
    pack = SMALL["p3_d64"]()
    # a negative lead
    bad_lead = pack.lead.copy()
    bad_lead[2] = -1
    got, err = run_kpool(cuda_lib, pack, False, lead=bad_lead, shift=shift)
    assert err == cuda_lib.CSA_DEVERR_LEAD
    assert (got == H.BF16_NAN).all()
    # more pools than out_rows
    got, err = run_kpool(cuda_lib, pack, False, out_rows=pack.total_pools - 1, shift=shift)
    assert err == cuda_lib.CSA_DEVERR_OUT_ROWS
    assert (got == H.BF16_NAN).all()
    # decreasing cu_seqlens
    cu = pack.cu_seqlens.copy()
    cu[2] = cu[1] - 1
    got, err = run_kpool(cuda_lib, pack, False, cu=cu, shift=shift)
    assert err == cuda_lib.CSA_DEVERR_CU_SEQLENS
    assert (got == H.BF16_NAN).all()


def test_kpool_no_pools(cuda_lib):
    """Segments that leave no complete pool (short, empty, lead past the end): no output
    row, no error."""
    pack = ts.make_kpool_custom([3, 0, 5, 2], pool=4, d=64, leads=[0, 0, 2, 9], seed=54)
    assert pack.total_pools == 0
    got, err = run_kpool(cuda_lib, pack, True, out_rows=0)
    assert err == 0
