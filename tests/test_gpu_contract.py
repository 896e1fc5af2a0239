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


def test_cuda_graph_capture_and_replay(cuda_lib):
    """fwd + bwd captured once in a CUDA graph and replayed on new inputs copied into the
    same buffers, with static-capacity padding rows (the graph case of the pages' zero
    ownership): every replay matches an eager call on the same inputs, bit for bit."""
    import torch
    a = ts.make_pack("ragged_r2_d512")
    b = ts.make_pack("ragged_r2_d512", seed=5)
    dev = H.device_pack(a)
    S, r, coff, d, cap, TC, C = a.S, a.ratio, a.coff, a.d, a.capacity, a.total_comp, a.C
    out = torch.empty((TC, d), dtype=torch.bfloat16, device="cuda")
    dkv = torch.empty((cap, C), dtype=torch.bfloat16, device="cuda")
    dsc = torch.empty_like(dkv)
    dape = torch.empty((r, C), dtype=torch.float32, device="cuda")
    wsb = cuda_lib.csa_compressor_bwd_workspace_bytes(S, r, coff, d, cap, TC)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")

    def step():
        cuda_lib.csa_compressor_fwd(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"], S, r,
                                    coff, d, cap, out, TC)
        cuda_lib.csa_compressor_bwd(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"],
                                    dev["dout"], S, r, coff, d, cap, TC, dkv, dsc, dape, 0, ws, wsb)

    step()  # first call on this device sets up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    for pack in (b, a, b):
        src = H.device_pack(pack)
        for k in ("kv", "score", "ape", "dout"):
            dev[k].copy_(src[k])
        dkv.view(torch.int16).fill_(np.int16(np.uint16(H.BF16_NAN).view(np.int16)))
        dsc.copy_(dkv)
        g.replay()
        torch.cuda.synchronize()
        got = (ts.bf16_tensor_bits(out), ts.bf16_tensor_bits(dkv), ts.bf16_tensor_bits(dsc),
               dape.cpu().numpy())
        ref_out, _ = H.run_fwd(cuda_lib, pack)
        rk, rs, rd, _ = H.run_bwd(cuda_lib, pack)
        assert (got[0] == ref_out).all() and (got[1] == rk).all() and (got[2] == rs).all()
        assert (got[3].view(np.uint32) == rd.view(np.uint32)).all()


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
