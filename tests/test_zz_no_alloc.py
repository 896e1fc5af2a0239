"""csa_compressor_bwd_noalloc: the backward for callers that cannot allocate device
memory (code inside allocator or memory-pool callbacks, plugins of hosts that own all
device memory). It uses the library's own file-scope device scratch array instead of a
caller workspace. Checked through the C ABI against csa_compressor_bwd on the same
inputs, on two calls in a row (the array keeps the previous call's contents), with the
output buffers pre-filled with NaN so that every element must be written.

This file is collected last on purpose, so that a run stopping at the first failure
has already run every other test.
"""
import numpy as np
import pytest

import thd_synth as ts
from tests import gpu_harness as H
from tests.parity import compare_bf16

pytestmark = pytest.mark.gpu


def _noalloc(gp, pack, dev, dape_init=None, accumulate=0):
    import torch
    C = pack.C
    fill = np.int16(np.uint16(H.BF16_NAN).view(np.int16))
    dkv = torch.full((pack.capacity, C), int(fill), dtype=torch.int16, device="cuda").view(torch.bfloat16)
    dsc = torch.full((pack.capacity, C), int(fill), dtype=torch.int16, device="cuda").view(torch.bfloat16)
    dape = torch.full((pack.ratio, C), float("nan"), dtype=torch.float32, device="cuda")
    if dape_init is not None:
        dape.copy_(torch.from_numpy(dape_init))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gp.csa_compressor_bwd_noalloc(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"],
                                  dev["dout"], pack.S, pack.ratio, pack.coff, pack.d,
                                  pack.capacity, pack.total_comp, dkv, dsc, dape, accumulate, err)
    torch.cuda.synchronize()
    return ts.bf16_tensor_bits(dkv), ts.bf16_tensor_bits(dsc), dape.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("name", ["3x8192_d512", "tiny"])
def test_noalloc_matches_workspace_entry_point(cuda_lib, name):
    pack = ts.make_pack(name)
    dev = H.device_pack(pack)
    ref_dkv, ref_dsc, ref_dape, err = H.run_bwd(cuda_lib, pack, dev=dev)
    assert err == 0
    for call in range(2):
        dkv, dsc, dape, err = _noalloc(cuda_lib, pack, dev)
        assert err == 0, (call, err)
        for label, got, ref in (("dkv", dkv, ref_dkv), ("dscore", dsc, ref_dsc)):
            rep = compare_bf16(label, got, ref)
            assert rep.fail == 0, (call, str(rep))
        np.testing.assert_allclose(dape, ref_dape, rtol=1e-5, atol=1e-6)
        # same kernels, same launch shape: the results are identical
        assert (dkv == ref_dkv).all() and (dsc == ref_dsc).all() and (dape == ref_dape).all()


def test_noalloc_rejects_sizes_beyond_the_scratch(cuda_lib):
    import torch
    # ratio=128 coff=1 d=512 with 40 output rows: the dAPE partials (one [128, 512] fp32
    # partial per row group) need more than the 4 MiB array
    pack = ts.make_custom([128] * 40, ratio=128, coff=1, d=512, pad_rows=0)
    need = cuda_lib.csa_compressor_bwd_workspace_bytes(pack.S, pack.ratio, pack.coff, pack.d,
                                                       pack.capacity, pack.total_comp)
    assert need > (4 << 20)
    dev = H.device_pack(pack)
    dkv = torch.empty((pack.capacity, pack.C), dtype=torch.bfloat16, device="cuda")
    dsc = torch.empty_like(dkv)
    dape = torch.empty((pack.ratio, pack.C), dtype=torch.float32, device="cuda")
    with pytest.raises(cuda_lib.CsaError) as ei:
        cuda_lib.csa_compressor_bwd_noalloc(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"],
                                            dev["dout"], pack.S, pack.ratio, pack.coff, pack.d,
                                            pack.capacity, pack.total_comp, dkv, dsc, dape, 0)
    assert ei.value.status == cuda_lib.CSA_ERR_UNSUPPORTED


def test_noalloc_rejected_call_leaves_dape_unchanged(cuda_lib):
    """After a valid call has left its dAPE partials in the shared scratch array, a call
    whose cu_seqlens the device rejects must not turn them into a dAPE: the caller's dAPE
    keeps its bits, with accumulate_dape=1 and =0."""
    import torch
    pack = ts.make_pack("tiny")
    dev = H.device_pack(pack)
    assert _noalloc(cuda_lib, pack, dev)[3] == 0
    bad = pack.cu_seqlens.copy()
    bad[2] = bad[1] - 1
    dev["cu_seqlens"] = torch.from_numpy(bad).cuda()
    base = np.linspace(-1, 1, pack.ratio * pack.C, dtype=np.float32).reshape(pack.ratio, pack.C)
    for acc in (1, 0):
        _, _, dape, err = _noalloc(cuda_lib, pack, dev, dape_init=base, accumulate=acc)
        assert err == cuda_lib.CSA_DEVERR_CU_SEQLENS
        assert (dape.view(np.uint32) == base.view(np.uint32)).all()
