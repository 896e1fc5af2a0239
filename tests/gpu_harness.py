"""Runs the CUDA library through its C ABI (Python binding) on a pack, for tests."""
import numpy as np

import thd_synth as ts

BF16_NAN = 0x7FC0


def device_pack(pack, shift=0):
    """The pack on the GPU; with shift > 0 every bf16/fp32 tensor starts `shift` elements
    past a 16-byte boundary (pointers the vector kernels cannot take)."""
    dev = ts.to_torch(pack, "cuda")
    if shift:
        dev = {k: (v if k == "cu_seqlens" else shifted_copy(v, shift)) for k, v in dev.items()}
    return dev


def shifted_empty(shape, dtype, shift):
    import torch
    n = 1
    for x in shape:
        n *= x
    if not shift:
        return torch.empty(shape, dtype=dtype, device="cuda")
    buf = torch.empty(n + 16, dtype=dtype, device="cuda")
    return buf[shift:shift + n].view(shape)


def shifted_copy(t, shift):
    v = shifted_empty(tuple(t.shape), t.dtype, shift)
    v.copy_(t)
    return v


def run_fwd(gp, pack, dev=None, out_rows=None, prefill_bits=None, stream=None, shift=0):
    import torch
    dev = dev or device_pack(pack, shift)
    out_rows = pack.total_comp if out_rows is None else out_rows
    out = shifted_empty((out_rows, pack.d), torch.int16, shift)
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
            accumulate=0, stream=None, dout=None, shift=0):
    import torch
    dev = dev or device_pack(pack, shift)
    out_rows = pack.total_comp if out_rows is None else out_rows
    C = pack.C
    fill = None if prefill_bits is None else np.int16(np.uint16(prefill_bits).view(np.int16))
    dkv = shifted_empty((pack.capacity, C), torch.int16, shift)
    dsc = shifted_empty((pack.capacity, C), torch.int16, shift)
    if fill is not None:
        dkv.fill_(fill)
        dsc.fill_(fill)
    dkv, dsc = dkv.view(torch.bfloat16), dsc.view(torch.bfloat16)
    dape = shifted_empty((pack.ratio, C), torch.float32, shift)
    dape.zero_()
    if dape_init is not None:
        dape.copy_(torch.from_numpy(dape_init))
    nbytes = gp.csa_compressor_bwd_workspace_bytes(pack.S, pack.ratio, pack.coff, pack.d,
                                                   pack.capacity, out_rows)
    ws = shifted_empty((max(nbytes, 16) // 4 + 4,), torch.float32, shift)
    if fill is not None:
        ws.fill_(float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if dout is None:
        dout = dev["dout"]
        if out_rows > pack.total_comp:  # pad dout rows that no block reads
            pad = torch.zeros((out_rows - pack.total_comp, pack.d), dtype=torch.bfloat16,
                              device="cuda")
            dout = torch.cat([dout, pad])
            if shift:
                dout = shifted_copy(dout, shift)
    gp.csa_compressor_bwd(dev["kv"], dev["score"], dev["ape"], dev["cu_seqlens"], dout,
                          pack.S, pack.ratio, pack.coff, pack.d, pack.capacity, out_rows, dkv,
                          dsc, dape, accumulate, ws, ws.numel() * 4, err, stream=stream)
    torch.cuda.synchronize()
    return (ts.bf16_tensor_bits(dkv), ts.bf16_tensor_bits(dsc), dape.cpu().numpy(),
            int(err.item()))
