"""ctypes front end of the fp64 CPU oracle (``csa_oracle.cpp``).

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package. The CUDA library never loads
it, and it never loads the CUDA library.

Arrays are numpy: bf16 tensors travel as their ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "libcsa_oracle.so")
_lib: Optional[ctypes.CDLL] = None

ERRORS = {0: "ok", 1: "bad arguments", 2: "invalid cu_seqlens", 3: "out_rows < total_comp",
          4: "a slot was read by two window positions", 5: "negative lead"}


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with g++ (plain -O2, no FMA contraction, no fast-math)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-shared",
           "-fPIC", "-pthread", "-o", out, src]
    subprocess.run(cmd, check=True)
    return out


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def load(path: Optional[str] = None) -> ctypes.CDLL:
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
    else:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.csa_oracle_total_comp.restype = i64
    lib.csa_oracle_total_comp.argtypes = [vp, i32, i32]
    lib.csa_oracle_map_blocks.restype = i32
    lib.csa_oracle_map_blocks.argtypes = [vp, i32, i32, i64, vp]
    lib.csa_oracle_fwd.restype = i32
    lib.csa_oracle_fwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i64, i64, vp, vp, vp]
    lib.csa_oracle_bwd.restype = i32
    lib.csa_oracle_bwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, i64,
                                   vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.csa_oracle_fwd_threads.restype = i32
    lib.csa_oracle_fwd_threads.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i64, i64, vp, i32]
    lib.csa_oracle_bwd_threads.restype = i32
    lib.csa_oracle_bwd_threads.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, i64,
                                           vp, vp, vp, i32]
    lib.csa_oracle_hardware_threads.restype = i32
    lib.csa_oracle_hardware_threads.argtypes = []
    lib.csa_oracle_round_bf16.restype = None
    lib.csa_oracle_round_bf16.argtypes = [vp, i64, vp]
    lib.csa_oracle_kpool_total.restype = i64
    lib.csa_oracle_kpool_total.argtypes = [vp, vp, i32, i32]
    lib.csa_oracle_kpool_fwd.restype = i32
    lib.csa_oracle_kpool_fwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i64, i64, i32, vp, vp, vp,
                                         vp, i32]
    if path is None:
        _lib = lib
    return lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"{what}: {ERRORS.get(rc, rc)}")


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def total_comp(cu_seqlens: np.ndarray, ratio: int, lib: Optional[ctypes.CDLL] = None) -> int:
    lib = lib or load()
    cu = _c(cu_seqlens, np.int32)
    n = int(lib.csa_oracle_total_comp(_p(cu), cu.shape[0] - 1, ratio))
    if n < 0:
        raise OracleError("total_comp: invalid cu_seqlens or ratio")
    return n


def map_blocks(cu_seqlens: np.ndarray, ratio: int, out_rows: int,
               lib: Optional[ctypes.CDLL] = None) -> np.ndarray:
    lib = lib or load()
    cu = _c(cu_seqlens, np.int32)
    out = np.empty((out_rows, 3), dtype=np.int32)
    _check(lib.csa_oracle_map_blocks(_p(cu), cu.shape[0] - 1, ratio, out_rows, _p(out)),
           "map_blocks")
    return out


def fwd(kv, score, ape, cu_seqlens, ratio: int, coff: int, d: int, capacity: int,
        out_rows: Optional[int] = None, *, want_f64: bool = False, want_err: bool = False,
        lib: Optional[ctypes.CDLL] = None) -> Dict[str, np.ndarray]:
    """Forward. Returns {"out": uint16 [out_rows, d], optional "out_f64", "out_err"}."""
    lib = lib or load()
    cu = _c(cu_seqlens, np.int32)
    if out_rows is None:
        out_rows = total_comp(cu, ratio, lib)
    kv, score, ape = _c(kv, np.uint16), _c(score, np.uint16), _c(ape, np.float32)
    res = {"out": np.zeros((out_rows, d), dtype=np.uint16)}
    if want_f64:
        res["out_f64"] = np.zeros((out_rows, d), dtype=np.float64)
    if want_err:
        res["out_err"] = np.zeros((out_rows, d), dtype=np.float64)
    _check(lib.csa_oracle_fwd(_p(kv), _p(score), _p(ape), _p(cu), cu.shape[0] - 1, ratio, coff,
                              d, capacity, out_rows, _p(res["out"]), _p(res.get("out_f64")),
                              _p(res.get("out_err"))), "fwd")
    return res


def bwd(kv, score, ape, cu_seqlens, dout, ratio: int, coff: int, d: int, capacity: int,
        out_rows: Optional[int] = None, *, want_f64: bool = False, want_owners: bool = False,
        want_err: bool = False, lib: Optional[ctypes.CDLL] = None) -> Dict[str, np.ndarray]:
    """Backward. Returns dkv/dscore (uint16 bf16 bits [capacity, coff*d]), dape_f64 and
    dape_f32 ([ratio, coff*d]); optionally the unrounded gradients, the per-slot owner
    counts and the error masses (dkv_err, dscore_err, dape_err; dape_abs)."""
    lib = lib or load()
    cu = _c(cu_seqlens, np.int32)
    if out_rows is None:
        out_rows = total_comp(cu, ratio, lib)
    C = coff * d
    kv, score, ape = _c(kv, np.uint16), _c(score, np.uint16), _c(ape, np.float32)
    dout = _c(dout, np.uint16) if dout is not None else None
    res = {
        "dkv": np.empty((capacity, C), dtype=np.uint16),
        "dscore": np.empty((capacity, C), dtype=np.uint16),
        "dape_f64": np.empty((ratio, C), dtype=np.float64),
        "dape_f32": np.empty((ratio, C), dtype=np.float32),
    }
    if want_f64:
        res["dkv_f64"] = np.empty((capacity, C), dtype=np.float64)
        res["dscore_f64"] = np.empty((capacity, C), dtype=np.float64)
    if want_owners:
        res["owners"] = np.empty((capacity, C), dtype=np.int32)
    if want_err:
        res["dkv_err"] = np.empty((capacity, C), dtype=np.float64)
        res["dscore_err"] = np.empty((capacity, C), dtype=np.float64)
        res["dape_err"] = np.empty((ratio, C), dtype=np.float64)
        res["dape_abs"] = np.empty((ratio, C), dtype=np.float64)
    _check(lib.csa_oracle_bwd(_p(kv), _p(score), _p(ape), _p(cu), _p(dout), cu.shape[0] - 1,
                              ratio, coff, d, capacity, out_rows, _p(res["dkv"]),
                              _p(res["dscore"]), _p(res["dape_f64"]), _p(res.get("dkv_f64")),
                              _p(res.get("dscore_f64")), _p(res["dape_f32"]),
                              _p(res.get("owners")), _p(res.get("dkv_err")),
                              _p(res.get("dscore_err")),
                              _p(res.get("dape_err")), _p(res.get("dape_abs"))), "bwd")
    return res


def hardware_threads(lib: Optional[ctypes.CDLL] = None) -> int:
    """Host threads the machine offers (std::thread::hardware_concurrency)."""
    return int((lib or load()).csa_oracle_hardware_threads())


def fwd_threads(pack, nthreads: int, lib: Optional[ctypes.CDLL] = None) -> np.ndarray:
    """Forward on ``nthreads`` host threads (output-row ranges); returns out bits."""
    lib = lib or load()
    cu = _c(pack.cu_seqlens, np.int32)
    kv, score, ape = _c(pack.kv, np.uint16), _c(pack.score, np.uint16), _c(pack.ape, np.float32)
    out = np.zeros((pack.total_comp, pack.d), dtype=np.uint16)
    _check(lib.csa_oracle_fwd_threads(_p(kv), _p(score), _p(ape), _p(cu), cu.shape[0] - 1,
                                      pack.ratio, pack.coff, pack.d, pack.capacity,
                                      pack.total_comp, _p(out), nthreads), "fwd_threads")
    return out


def bwd_threads(pack, nthreads: int, lib: Optional[ctypes.CDLL] = None) -> Dict[str, np.ndarray]:
    """Backward on ``nthreads`` host threads; returns dkv, dscore bits and dape_f64."""
    lib = lib or load()
    cu = _c(pack.cu_seqlens, np.int32)
    kv, score, ape = _c(pack.kv, np.uint16), _c(pack.score, np.uint16), _c(pack.ape, np.float32)
    dout = _c(pack.dout, np.uint16)
    C = pack.coff * pack.d
    res = {"dkv": np.empty((pack.capacity, C), dtype=np.uint16),
           "dscore": np.empty((pack.capacity, C), dtype=np.uint16),
           "dape_f64": np.empty((pack.ratio, C), dtype=np.float64)}
    _check(lib.csa_oracle_bwd_threads(_p(kv), _p(score), _p(ape), _p(cu), _p(dout),
                                      cu.shape[0] - 1, pack.ratio, pack.coff, pack.d,
                                      pack.capacity, pack.total_comp, _p(res["dkv"]),
                                      _p(res["dscore"]), _p(res["dape_f64"]), nthreads),
           "bwd_threads")
    return res


def round_bf16(x: np.ndarray, lib: Optional[ctypes.CDLL] = None) -> np.ndarray:
    lib = lib or load()
    x = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.csa_oracle_round_bf16(_p(x), x.size, _p(out))
    return out


def fwd_pack(pack, **kw):
    return fwd(pack.kv, pack.score, pack.ape, pack.cu_seqlens, pack.ratio, pack.coff, pack.d,
               pack.capacity, **kw)


def bwd_pack(pack, **kw):
    return bwd(pack.kv, pack.score, pack.ape, pack.cu_seqlens, pack.dout, pack.ratio, pack.coff,
               pack.d, pack.capacity, **kw)


# ----------------------------------------------------------------------------------
# KPool (the DSA indexer's key pooling)
# ----------------------------------------------------------------------------------

def kpool_total(cu_seqlens, lead, pool: int, lib: Optional[ctypes.CDLL] = None) -> int:
    """Number of pools: sum over segments of floor((seqlen - lead) / pool)."""
    lib = lib or load()
    cu = _c(cu_seqlens, np.int32)
    ld = None if lead is None else _c(lead, np.int32)
    n = lib.csa_oracle_kpool_total(_p(cu), _p(ld), cu.shape[0] - 1, pool)
    if n < 0:
        raise OracleError("kpool_total: bad arguments")
    return int(n)


def kpool_fwd(key, gate, cu_seqlens, lead, pool: int, d: int, capacity: int,
              out_rows: Optional[int] = None, *, compress: bool = False, want_f64: bool = False,
              want_err: bool = False, nthreads: int = 1,
              lib: Optional[ctypes.CDLL] = None) -> Dict[str, np.ndarray]:
    """KPool forward. Returns {"out": uint16 [out_rows, d], optional "out_f64", "out_err"
    and "out_slack" (the last two with want_err)}."""
    lib = lib or load()
    cu = _c(cu_seqlens, np.int32)
    ld = None if lead is None else _c(lead, np.int32)
    if out_rows is None:
        out_rows = kpool_total(cu, ld, pool, lib)
    key, gate = _c(key, np.uint16), _c(gate, np.uint16)
    res = {"out": np.zeros((out_rows, d), dtype=np.uint16)}
    if want_f64:
        res["out_f64"] = np.zeros((out_rows, d), dtype=np.float64)
    if want_err:
        res["out_err"] = np.zeros((out_rows, d), dtype=np.float64)
        res["out_slack"] = np.zeros((out_rows, d), dtype=np.float64)
    _check(lib.csa_oracle_kpool_fwd(_p(key), _p(gate), _p(cu), _p(ld), cu.shape[0] - 1, pool, d,
                                    capacity, out_rows, 1 if compress else 0, _p(res["out"]),
                                    _p(res.get("out_f64")), _p(res.get("out_err")),
                                    _p(res.get("out_slack")), max(1, nthreads)), "kpool_fwd")
    return res


def kpool_fwd_pack(pack, **kw):
    return kpool_fwd(pack.key, pack.gate, pack.cu_seqlens, pack.lead, pack.pool, pack.d,
                     pack.capacity, **kw)

