"""Runs the CUDA library through its C ABI (Python binding) on a pack, for tests."""
import numpy as np

import thd_synth as ts

BF16_NAN = 0x7FC0


def device_pack(pack):
    return ts.to_torch(pack, "cuda")


def run_fwd(gp, pack, dev=None, out_rows=None, prefill_bits=None, stream=None):
    import torch
    dev = dev or device_pack(pack)
    out_rows = pack.total_comp if out_rows is None else out_rows
    out = torch.empty((out_rows, pack.d), dtype=torch.int16, device="cuda")
    if prefill_bits is not None:
        out.fill_(np.int16(np.uint16(prefill_bits).view(np.int16)))
    out = out.view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gp.csa_compressor_fwd(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"], pack.S,
                          pack.ratio, pack.coff, pack.d, pack.capacity, out, out_rows, err,
                          stream=stream)
    torch.cuda.synchronize()
    return ts.bf16_tensor_bits(out), int(err.item())


def run_bwd(gp, pack, dev=None, out_rows=None, prefill_bits=None, dape_init=None,
            accumulate=0, stream=None, dout=None):
    import torch
    dev = dev or device_pack(pack)
    out_rows = pack.total_comp if out_rows is None else out_rows
    C = pack.C
    fill = None if prefill_bits is None else np.int16(np.uint16(prefill_bits).view(np.int16))
    dkv = torch.empty((pack.capacity, C), dtype=torch.int16, device="cuda")
    dsc = torch.empty((pack.capacity, C), dtype=torch.int16, device="cuda")
    if fill is not None:
        dkv.fill_(fill)
        dsc.fill_(fill)
    dkv, dsc = dkv.view(torch.bfloat16), dsc.view(torch.bfloat16)
    dape = torch.zeros((pack.ratio, C), dtype=torch.float32, device="cuda")
    if dape_init is not None:
        dape.copy_(torch.from_numpy(dape_init))
    nbytes = gp.csa_compressor_bwd_workspace_bytes(pack.S, pack.ratio, pack.coff, pack.d,
                                                   pack.capacity, out_rows)
    ws = torch.empty(max(nbytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")
    if fill is not None:
        ws.fill_(float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if dout is None:
        dout = dev["dout"]
        if out_rows > pack.total_comp:  # pad dout rows that no block reads
            pad = torch.zeros((out_rows - pack.total_comp, pack.d), dtype=torch.bfloat16,
                              device="cuda")
            dout = torch.cat([dout, pad])
    gp.csa_compressor_bwd(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"], dout,
                          pack.S, pack.ratio, pack.coff, pack.d, pack.capacity, out_rows, dkv,
                          dsc, dape, accumulate, ws, ws.numel() * 4, err, stream=stream)
    torch.cuda.synchronize()
    return (ts.bf16_tensor_bits(dkv), ts.bf16_tensor_bits(dsc), dape.cpu().numpy(),
            int(err.item()))
