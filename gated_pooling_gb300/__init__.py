"""GB300 (sm_103a) CSA/HCA KV-compressor gated-softmax pooling over THD packs.

A thin ctypes binding of the C ABI in ``include/csa_compressor.h``: the functions
below have the C names and arguments, and only marshal them (tensor -> device
pointer, stream -> cudaStream_t). Every step of the pooling runs in the library's
CUDA kernels. There is no fallback: if the library is missing, loading raises.

Tensors are torch CUDA tensors (bf16 for kv/score/dout/out/dkv/dscore and the KPool
key/gate, fp32 for ape/dape, int32 for cu_seqlens, lead and the error word); PyTorch
only provides device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

LIB_PATH = _build.LIB
_lib: Optional[ctypes.CDLL] = None

CSA_OK, CSA_ERR_INVALID_VALUE, CSA_ERR_UNSUPPORTED, CSA_ERR_WORKSPACE, CSA_ERR_CUDA = 0, 1, 2, 3, 4
CSA_DEVERR_CU_SEQLENS, CSA_DEVERR_OUT_ROWS, CSA_DEVERR_TIMEOUT, CSA_DEVERR_LEAD = 1, 2, 3, 4
CSA_TEST_MIN_WAIT_CYCLES = 1000000
CSA_KPOOL_MAX_POOL = 1024
EXPORTED = ("csa_status_string", "csa_last_error_string", "csa_compressor_total_comp", "csa_compressor_fwd",
            "csa_compressor_bwd_workspace_bytes", "csa_compressor_bwd",
            "csa_compressor_bwd_noalloc", "csa_compressor_test_hooks",
            "csa_compressor_map_blocks", "csa_kpool_total", "csa_kpool_fwd")


class CsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads the CUDA library (building it first only if ``path`` is None and it is
    missing or stale). Raises if it cannot be loaded."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    if path is None:
        if not _build.up_to_date():
            _build.build()
        path = LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not found at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.csa_status_string.restype = ctypes.c_char_p
    lib.csa_status_string.argtypes = [ctypes.c_int]
    lib.csa_last_error_string.restype = ctypes.c_char_p
    lib.csa_last_error_string.argtypes = []
    lib.csa_compressor_total_comp.restype = i64
    lib.csa_compressor_total_comp.argtypes = [vp, i32, i32]
    lib.csa_compressor_fwd.restype = ctypes.c_int
    lib.csa_compressor_fwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i64, vp, i64, vp, vp]
    lib.csa_compressor_bwd_workspace_bytes.restype = sz
    lib.csa_compressor_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32, i64, i64]
    lib.csa_compressor_bwd.restype = ctypes.c_int
    lib.csa_compressor_bwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, i64, vp, vp,
                                       vp, i32, vp, sz, vp, vp]
    lib.csa_compressor_bwd_noalloc.restype = ctypes.c_int
    lib.csa_compressor_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, i64,
                                               vp, vp, vp, i32, vp, vp]
    lib.csa_compressor_test_hooks.restype = ctypes.c_int
    lib.csa_compressor_test_hooks.argtypes = [i64, i32]
    lib.csa_compressor_map_blocks.restype = ctypes.c_int
    lib.csa_compressor_map_blocks.argtypes = [vp, i32, i32, i64, i64, vp, vp, vp]
    lib.csa_kpool_total.restype = i64
    lib.csa_kpool_total.argtypes = [vp, vp, i32, i32]
    lib.csa_kpool_fwd.restype = ctypes.c_int
    lib.csa_kpool_fwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i64, vp, i64, i32, vp, vp]
    if path == LIB_PATH:
        _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != CSA_OK:
        msg = load().csa_status_string(status).decode()
        if status == CSA_ERR_CUDA:
            msg += f" ({load().csa_last_error_string().decode()})"
        raise CsaError(status, f"{what}: {msg}")


def csa_status_string(status: int) -> str:
    return load().csa_status_string(status).decode()


def csa_last_error_string() -> str:
    return load().csa_last_error_string().decode()


def csa_compressor_total_comp(cu_seqlens_host, S: int, ratio: int) -> int:
    """``cu_seqlens_host``: a host int32 array (numpy, CPU tensor or ctypes pointer)."""
    import numpy as np
    if hasattr(cu_seqlens_host, "numpy"):
        cu_seqlens_host = cu_seqlens_host.numpy()
    arr = np.ascontiguousarray(cu_seqlens_host, dtype=np.int32)
    return int(load().csa_compressor_total_comp(arr.ctypes.data_as(ctypes.c_void_p), S, ratio))


def csa_compressor_fwd(kv, score, ape, cu_seqlens, S: int, ratio: int, coff: int, d: int,
                       capacity: int, out, out_rows: int, dev_error=None, stream=None) -> None:
    _check(load().csa_compressor_fwd(_ptr(kv), _ptr(score), _ptr(ape), _ptr(cu_seqlens), S,
                                     ratio, coff, d, capacity, _ptr(out), out_rows,
                                     _ptr(dev_error), _stream(stream)), "csa_compressor_fwd")


def csa_compressor_bwd_workspace_bytes(S: int, ratio: int, coff: int, d: int, capacity: int,
                                       out_rows: int) -> int:
    return int(load().csa_compressor_bwd_workspace_bytes(S, ratio, coff, d, capacity, out_rows))


def csa_compressor_bwd(kv, score, ape, cu_seqlens, dout, S: int, ratio: int, coff: int, d: int,
                       capacity: int, out_rows: int, dkv, dscore, dape, accumulate_dape: int,
                       workspace, workspace_bytes: int, dev_error=None, stream=None) -> None:
    _check(load().csa_compressor_bwd(_ptr(kv), _ptr(score), _ptr(ape), _ptr(cu_seqlens),
                                     _ptr(dout), S, ratio, coff, d, capacity, out_rows, _ptr(dkv),
                                     _ptr(dscore), _ptr(dape), int(accumulate_dape),
                                     _ptr(workspace), workspace_bytes, _ptr(dev_error),
                                     _stream(stream)), "csa_compressor_bwd")


def csa_compressor_bwd_noalloc(kv, score, ape, cu_seqlens, dout, S: int, ratio: int, coff: int,
                               d: int, capacity: int, out_rows: int, dkv, dscore, dape,
                               accumulate_dape: int, dev_error=None, stream=None) -> None:
    """Backward without a caller workspace, for callers that cannot allocate device
    memory; see include/csa_compressor.h for the shared scratch array's rules."""
    _check(load().csa_compressor_bwd_noalloc(_ptr(kv), _ptr(score), _ptr(ape), _ptr(cu_seqlens),
                                             _ptr(dout), S, ratio, coff, d, capacity, out_rows,
                                             _ptr(dkv), _ptr(dscore), _ptr(dape),
                                             int(accumulate_dape), _ptr(dev_error),
                                             _stream(stream)), "csa_compressor_bwd_noalloc")


def csa_compressor_test_hooks(wait_cycles: int, withhold_row: int) -> None:
    """Test hook: pipeline wait bound (0 = default) and the row whose copies the first
    CTA's producer withholds (-1 = off), for every later call."""
    _check(load().csa_compressor_test_hooks(int(wait_cycles), int(withhold_row)),
           "csa_compressor_test_hooks")


def csa_compressor_map_blocks(cu_seqlens, S: int, ratio: int, capacity: int, out_rows: int,
                              seg_blk_base, dev_error=None, stream=None) -> None:
    _check(load().csa_compressor_map_blocks(_ptr(cu_seqlens), S, ratio, capacity, out_rows,
                                            _ptr(seg_blk_base), _ptr(dev_error),
                                            _stream(stream)), "csa_compressor_map_blocks")


def csa_kpool_total(cu_seqlens_host, lead_host, S: int, pool: int) -> int:
    """Pool count from host int32 arrays (``lead_host`` may be None)."""
    import numpy as np
    def arr(x):
        if x is None:
            return None
        if hasattr(x, "numpy"):
            x = x.numpy()
        return np.ascontiguousarray(x, dtype=np.int32)
    cu, ld = arr(cu_seqlens_host), arr(lead_host)
    return int(load().csa_kpool_total(cu.ctypes.data_as(ctypes.c_void_p),
                                      None if ld is None else ld.ctypes.data_as(ctypes.c_void_p),
                                      S, pool))


def csa_kpool_fwd(key, gate, cu_seqlens, lead, S: int, pool: int, d: int, capacity: int, out,
                  out_rows: int, compress: int = 0, dev_error=None, stream=None) -> None:
    """KPool forward (the DSA indexer's key pooling); ``lead`` may be None."""
    _check(load().csa_kpool_fwd(_ptr(key), _ptr(gate), _ptr(cu_seqlens), _ptr(lead), S, pool, d,
                                capacity, _ptr(out), out_rows, int(compress), _ptr(dev_error),
                                _stream(stream)), "csa_kpool_fwd")

