"""Buffer contract and robustness of the CUDA path, through the C ABI.

* run-to-run determinism: out, dKV, dScore and dAPE are bitwise identical across runs
  (the pages guarantee it for out/dKV/dScore; here dAPE too, since nothing is atomic);
* NaN canary: outputs pre-filled with NaN come back bitwise identical to outputs
  pre-filled with zeros (every position is written, "fold dKV/dScore zero-init into the
  backward kernel", Megatron-LM PR #5984);
* guard bands: nothing outside the output buffers is touched;
* device-detected errors: bad cu_seqlens and too few out_rows set the error word and
  leave the outputs unwritten;
* accumulate_dape adds to the current dAPE; a non-default stream works; out_rows larger
  than total_comp leaves the extra rows untouched;
* a call reads what the previous call on its stream wrote (programmatic launch);
* fwd + bwd captured in a CUDA graph replay bit for bit on new inputs.
"""
import numpy as np
import pytest

import thd_synth as ts
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

PACKS = ["tiny", "ragged_r2_d512", "long_r128_d512"]


def _pack(name):
    if name == "many":
        return ts.make_custom(list(np.random.default_rng(4).integers(0, 30, 300)), ratio=4, coff=2,
                              d=64, pad_rows=17, seed=3)
    return ts.make_pack(name)


@pytest.mark.parametrize("name", PACKS + ["many"])
def test_bitwise_deterministic_and_nan_canary(cuda_lib, name):
    pack = _pack(name)
    dev = H.device_pack(pack)
    f1, e1 = H.run_fwd(cuda_lib, pack, dev=dev, prefill_bits=H.BF16_NAN)
    f2, e2 = H.run_fwd(cuda_lib, pack, dev=dev, prefill_bits=0)
    assert e1 == e2 == 0
    assert (f1 == f2).all()
    a = H.run_bwd(cuda_lib, pack, dev=dev, prefill_bits=H.BF16_NAN)
    b = H.run_bwd(cuda_lib, pack, dev=dev, prefill_bits=0)
    c = H.run_bwd(cuda_lib, pack, dev=dev)
    for x, y in ((a, b), (b, c)):
        assert x[3] == y[3] == 0
        assert (x[0] == y[0]).all() and (x[1] == y[1]).all()
        assert (x[2].view(np.uint32) == y[2].view(np.uint32)).all()


def test_guard_bands_untouched(cuda_lib):
    import torch
    pack = ts.make_pack("tiny")
    dev = H.device_pack(pack)
    G = 4096  # guard elements on each side
    C, cap, TC, d = pack.C, pack.capacity, pack.total_comp, pack.d
    sentinel = np.int16(0x5A5A)

    def guarded(n):
        buf = torch.full((n + 2 * G,), int(sentinel), dtype=torch.int16, device="cuda")
        return buf, buf[G:G + n].view(torch.bfloat16)

    ob, out = guarded(TC * d)
    kb, dkv = guarded(cap * C)
    sb, dsc = guarded(cap * C)
    ab = torch.full((pack.ratio * C + 2 * G,), 7.0, dtype=torch.float32, device="cuda")
    dape = ab[G:G + pack.ratio * C]
    nbytes = cuda_lib.csa_compressor_bwd_workspace_bytes(pack.S, pack.ratio, pack.coff, d, cap, TC)
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device="cuda")
    cuda_lib.csa_compressor_fwd(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"], pack.S,
                                pack.ratio, pack.coff, d, cap, out, TC)
    cuda_lib.csa_compressor_bwd(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"], dev["dout"],
                                pack.S, pack.ratio, pack.coff, d, cap, TC, dkv, dsc, dape, 0, ws,
                                ws.numel() * 4)
    torch.cuda.synchronize()
    for buf, n in ((ob, TC * d), (kb, cap * C), (sb, cap * C)):
        h = buf.cpu().numpy()
        assert (h[:G] == sentinel).all() and (h[G + n:] == sentinel).all()
    h = ab.cpu().numpy()
    assert (h[:G] == 7.0).all() and (h[G + pack.ratio * C:] == 7.0).all()


def test_device_error_bad_cu_seqlens(cuda_lib):
    import torch
    pack = ts.make_pack("tiny")
    dev = H.device_pack(pack)
    bad = pack.cu_seqlens.copy()
    bad[2] = bad[1] - 1                         # decreasing
    dev["cu_seqlens"] = torch.from_numpy(bad).cuda()
    out, err = H.run_fwd(cuda_lib, pack, dev=dev, prefill_bits=0x1234)
    assert err == cuda_lib.CSA_DEVERR_CU_SEQLENS
    assert (out == 0x1234).all()                # nothing written
    dkv, dsc, dape, err = H.run_bwd(cuda_lib, pack, dev=dev, prefill_bits=0x1234)
    assert err == cuda_lib.CSA_DEVERR_CU_SEQLENS
    assert (dkv == 0x1234).all() and (dsc == 0x1234).all()
    past = pack.cu_seqlens.copy()
    past[-1] = pack.capacity + 1                # past capacity
    dev["cu_seqlens"] = torch.from_numpy(past).cuda()
    out, err = H.run_fwd(cuda_lib, pack, dev=dev, out_rows=pack.total_comp + 1, prefill_bits=0x1234)
    assert err == cuda_lib.CSA_DEVERR_CU_SEQLENS


def test_rejected_call_leaves_dape_unchanged(cuda_lib):
    """A backward whose cu_seqlens the device rejects writes no output at all: with
    accumulate_dape=1 (and =0) the caller's dAPE keeps its bits, also after a valid call
    has left its partials in the same workspace."""
    import torch
    pack = ts.make_pack("tiny")
    dev = H.device_pack(pack)
    H.run_bwd(cuda_lib, pack, dev=dev)  # a valid call first
    bad = pack.cu_seqlens.copy()
    bad[2] = bad[1] - 1
    dev["cu_seqlens"] = torch.from_numpy(bad).cuda()
    base = np.linspace(-1, 1, pack.ratio * pack.C, dtype=np.float32).reshape(pack.ratio, pack.C)
    for acc in (1, 0):
        _, _, dape, err = H.run_bwd(cuda_lib, pack, dev=dev, dape_init=base, accumulate=acc)
        assert err == cuda_lib.CSA_DEVERR_CU_SEQLENS
        assert (dape.view(np.uint32) == base.view(np.uint32)).all()


def test_device_error_out_rows_too_small(cuda_lib):
    pack = ts.make_pack("tiny")
    out, err = H.run_fwd(cuda_lib, pack, out_rows=pack.total_comp - 1, prefill_bits=0x1234)
    assert err == cuda_lib.CSA_DEVERR_OUT_ROWS
    assert (out == 0x1234).all()


def test_out_rows_slack_untouched(cuda_lib):
    pack = ts.make_pack("ragged_r2_d512")
    extra = 5
    out, err = H.run_fwd(cuda_lib, pack, out_rows=pack.total_comp + extra, prefill_bits=0x1234)
    assert err == 0
    ref, _ = H.run_fwd(cuda_lib, pack)
    out = out.reshape(-1, pack.d)
    assert (out[pack.total_comp:] == 0x1234).all()
    assert (out[:pack.total_comp] == ref.reshape(-1, pack.d)).all()
    a = H.run_bwd(cuda_lib, pack, out_rows=pack.total_comp + extra)
    b = H.run_bwd(cuda_lib, pack)
    assert a[3] == 0 and (a[0] == b[0]).all() and (a[1] == b[1]).all()


def test_accumulate_dape(cuda_lib):
    pack = ts.make_pack("tiny")
    base = np.linspace(-1, 1, pack.ratio * pack.C, dtype=np.float32).reshape(pack.ratio, pack.C)
    _, _, d0, _ = H.run_bwd(cuda_lib, pack)
    _, _, d1, _ = H.run_bwd(cuda_lib, pack, dape_init=base, accumulate=1)
    np.testing.assert_allclose(d1, base + d0, rtol=1e-6, atol=1e-7)


def test_non_default_stream(cuda_lib):
    import torch
    pack = ts.make_pack("1x8192_d128")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a, e = H.run_fwd(cuda_lib, pack, stream=s)
    b, _ = H.run_fwd(cuda_lib, pack)
    assert e == 0 and (a == b).all()


def _graph_packs():
    """Two ragged ratio=2 coff=2 d=64 packs with the same segment count and token capacity
    (static-capacity padding: 300 and 399 rows past cu_seqlens[S]), short and empty
    segments, different lengths and values."""
    a = ts.make_custom([700, 1, 3, 513, 0, 800], ratio=2, coff=2, d=64, pad_rows=300, seed=50)
    b = ts.make_custom([300, 2, 900, 11, 5, 700], ratio=2, coff=2, d=64, pad_rows=399, seed=51)
    assert a.capacity == b.capacity and a.S == b.S
    return a, b


def test_cuda_graph_capture_and_replay(cuda_lib):
    """fwd + bwd captured once in a CUDA graph and replayed on new inputs (other values
    and other segment lengths) copied into the same buffers, with static-capacity padding
    rows (the graph case of the pages' zero ownership, "Megatron-LM PR #5984", commits
    "CSA: add fused Compressor..." and "fold dKV/dScore zero-init into the backward
    kernel"): every replay, with its gradient buffers pre-filled with NaN, matches the
    fp64 oracle on that replay's inputs under the parity tolerance."""
    import torch
    from tests.parity import compare_bf16, compare_dape
    import oracle

    a, b = _graph_packs()
    S, r, coff, d, cap, C = a.S, a.ratio, a.coff, a.d, a.capacity, a.C
    rows = max(a.total_comp, b.total_comp)  # out_rows: room for either pack's blocks
    dev = H.device_pack(a)
    dev["dout"] = torch.zeros((rows, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((rows, d), dtype=torch.bfloat16, device="cuda")
    dkv = torch.empty((cap, C), dtype=torch.bfloat16, device="cuda")
    dsc = torch.empty_like(dkv)
    dape = torch.empty((r, C), dtype=torch.float32, device="cuda")
    wsb = cuda_lib.csa_compressor_bwd_workspace_bytes(S, r, coff, d, cap, rows)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        cuda_lib.csa_compressor_fwd(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"], S, r,
                                    coff, d, cap, out, rows, err)
        cuda_lib.csa_compressor_bwd(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"],
                                    dev["dout"], S, r, coff, d, cap, rows, dkv, dsc, dape, 0, ws,
                                    wsb, err)

    step()  # first call on this device sets up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    nan = np.int16(np.uint16(H.BF16_NAN).view(np.int16))
    for pack in (b, a, b):
        src = H.device_pack(pack)
        for k in ("kv", "score", "ape", "cu_seqlens"):
            dev[k].copy_(src[k])
        dev["dout"].zero_()
        dev["dout"][:pack.total_comp].copy_(src["dout"])
        dkv.view(torch.int16).fill_(nan)
        dsc.view(torch.int16).fill_(nan)
        dape.fill_(float("nan"))
        err.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        TC = pack.total_comp
        ref = oracle.fwd_pack(pack, want_f64=True, want_err=True)
        refb = oracle.bwd_pack(pack, want_f64=True, want_err=True, want_owners=True)
        got_out = ts.bf16_tensor_bits(out[:TC])
        got_dkv, got_dsc = ts.bf16_tensor_bits(dkv), ts.bf16_tensor_bits(dsc)
        reps = (compare_bf16("out", got_out, ref["out"], ref["out_f64"], ref["out_err"]),
                compare_bf16("dkv", got_dkv, refb["dkv"], refb["dkv_f64"], refb["dkv_err"]),
                compare_bf16("dscore", got_dsc, refb["dscore"], refb["dscore_f64"],
                             refb["dscore_err"]),
                compare_dape(dape.cpu().numpy(), refb["dape_f64"], refb["dape_err"]))
        for rep in reps:
            assert rep.fail == 0, str(rep)
        zero = refb["owners"] == 0
        assert (got_dkv.reshape(zero.shape)[zero] == 0).all()
        assert (got_dsc.reshape(zero.shape)[zero] == 0).all()


def test_back_to_back_calls_see_previous_results(cuda_lib):
    """Every call is launched as a programmatic dependent of the stream's previous kernel,
    so it may start before that kernel ends; it must still read that kernel's results. A
    forward call writes its output into a NaN-filled buffer which the next forward call
    (ratio 1, coff 1: its output is its kv) reads as kv and score, back to back on one
    stream: the second output must equal the first, bit for bit, every time."""
    import torch
    a = ts.make_custom([65536], ratio=2, coff=1, d=512, pad_rows=0, seed=40)
    dev = H.device_pack(a)
    T2, d = a.total_comp, a.d
    ref, _ = H.run_fwd(cuda_lib, a)
    ape1 = torch.zeros((1, d), dtype=torch.float32, device="cuda")
    cu1 = torch.tensor([0, T2], dtype=torch.int32, device="cuda")
    x = torch.empty((T2, d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T2, d), dtype=torch.bfloat16, device="cuda")
    nan = np.int16(np.uint16(H.BF16_NAN).view(np.int16))
    for _ in range(5):
        x.view(torch.int16).fill_(nan)
        y.view(torch.int16).fill_(nan)
        cuda_lib.csa_compressor_fwd(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"], a.S,
                                    a.ratio, a.coff, d, a.capacity, x, T2)
        cuda_lib.csa_compressor_fwd(x, x, ape1, cu1, 1, 1, 1, d, T2, y, T2)
        torch.cuda.synchronize()
        assert (ts.bf16_tensor_bits(x) == ref).all()
        assert (ts.bf16_tensor_bits(y) == ref).all()
