"""The C-ABI library builds, loads and exports every entry point its header declares;
host-side argument checks return the documented status codes. CPU only: no call
here reaches the GPU (every call is rejected before any CUDA runtime call)."""
import ctypes
import os
import re

import numpy as np
import pytest

import gated_pooling_gb300 as gp
import oracle

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "csa_compressor.h")


@pytest.fixture(scope="module")
def lib():
    return gp.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\S[^\n(]*?\b(csa_\w+)\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(gp.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(5):
        assert gp.csa_status_string(code).startswith("CSA_")
    assert gp.csa_status_string(gp.CSA_ERR_WORKSPACE).startswith("CSA_ERR_WORKSPACE")
    assert gp.csa_status_string(gp.CSA_ERR_CUDA).startswith("CSA_ERR_CUDA")


def test_status_codes_match_header():
    text = open(HEADER).read()
    for name in ("CSA_OK", "CSA_ERR_INVALID_VALUE", "CSA_ERR_UNSUPPORTED", "CSA_ERR_WORKSPACE",
                 "CSA_ERR_CUDA"):
        m = re.search(rf"\b{name} = (\d+)", text)
        assert m and int(m.group(1)) == getattr(gp, name), name
    for name in ("CSA_DEVERR_CU_SEQLENS", "CSA_DEVERR_OUT_ROWS", "CSA_DEVERR_TIMEOUT",
                 "CSA_DEVERR_LEAD", "CSA_TEST_MIN_WAIT_CYCLES", "CSA_KPOOL_MAX_POOL"):
        m = re.search(rf"#define {name} (\d+)", text)
        assert m and int(m.group(1)) == getattr(gp, name), name


def test_total_comp_host_helper(lib, oracle_lib):
    rng = np.random.default_rng(0)
    for _ in range(50):
        S = int(rng.integers(0, 9))
        cu = np.concatenate([[0], np.cumsum(rng.integers(0, 40, S))]).astype(np.int32)
        r = int(rng.integers(1, 9))
        assert gp.csa_compressor_total_comp(cu, S, r) == oracle.total_comp(cu, r)
    assert gp.csa_compressor_total_comp(np.array([0, 5, 3], np.int32), 2, 2) == -1
    assert gp.csa_compressor_total_comp(np.array([0], np.int32), 0, 0) == -1


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced (calls are rejected)


def fwd_status(lib, **over):
    a = dict(kv=FAKE, score=FAKE, ape=FAKE, cu=FAKE, S=1, ratio=4, coff=2, d=8, capacity=8,
             out=FAKE, out_rows=2, err=None)
    a.update(over)
    return lib.csa_compressor_fwd(a["kv"], a["score"], a["ape"], a["cu"], a["S"], a["ratio"],
                                  a["coff"], a["d"], a["capacity"], a["out"], a["out_rows"],
                                  a["err"], None)


def bwd_status(lib, **over):
    a = dict(kv=FAKE, score=FAKE, ape=FAKE, cu=FAKE, dout=FAKE, S=1, ratio=4, coff=2, d=8,
             capacity=8, out_rows=2, dkv=FAKE, dscore=FAKE, dape=FAKE, acc=0, ws=FAKE,
             ws_bytes=1 << 20, err=None)
    a.update(over)
    return lib.csa_compressor_bwd(a["kv"], a["score"], a["ape"], a["cu"], a["dout"], a["S"],
                                  a["ratio"], a["coff"], a["d"], a["capacity"], a["out_rows"],
                                  a["dkv"], a["dscore"], a["dape"], a["acc"], a["ws"],
                                  a["ws_bytes"], a["err"], None)


@pytest.mark.parametrize("over,code", [
    (dict(coff=0), gp.CSA_ERR_UNSUPPORTED),
    (dict(coff=3), gp.CSA_ERR_UNSUPPORTED),
    (dict(d=12, ratio=200), gp.CSA_ERR_UNSUPPORTED),  # d % 8 != 0: generic, window 400 > 256
    (dict(S=20000), gp.CSA_ERR_UNSUPPORTED),
    (dict(ratio=2048), gp.CSA_ERR_UNSUPPORTED),          # window 4096 > 2048
    (dict(capacity=1 << 28, d=64), gp.CSA_ERR_UNSUPPORTED),  # capacity*coff*d >= 2^31
    (dict(out_rows=1 << 28, d=64), gp.CSA_ERR_UNSUPPORTED),
    (dict(S=-1), gp.CSA_ERR_INVALID_VALUE),
    (dict(ratio=0), gp.CSA_ERR_INVALID_VALUE),
    (dict(d=0), gp.CSA_ERR_INVALID_VALUE),
    (dict(capacity=-1), gp.CSA_ERR_INVALID_VALUE),
    (dict(out_rows=-1), gp.CSA_ERR_INVALID_VALUE),
    (dict(cu=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(ape=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(kv=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(out=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(kv=FAKE + 1), gp.CSA_ERR_INVALID_VALUE),      # misaligned for bf16
    (dict(ape=FAKE + 2), gp.CSA_ERR_INVALID_VALUE),     # misaligned for fp32
    (dict(out=FAKE + 1), gp.CSA_ERR_INVALID_VALUE),
    (dict(out=FAKE + 2, ratio=200), gp.CSA_ERR_UNSUPPORTED),  # unaligned: generic, window too long
])
def test_fwd_rejects(lib, over, code):
    assert fwd_status(lib, **over) == code


@pytest.mark.parametrize("over,code", [
    (dict(coff=3), gp.CSA_ERR_UNSUPPORTED),
    (dict(d=4, ratio=129), gp.CSA_ERR_UNSUPPORTED),  # generic, window 258 > 256
    (dict(dape=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(dkv=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(dscore=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(dout=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(dscore=FAKE + 1), gp.CSA_ERR_INVALID_VALUE),
    (dict(dape=FAKE + 2), gp.CSA_ERR_INVALID_VALUE),
    (dict(ws=FAKE + 2), gp.CSA_ERR_INVALID_VALUE),
    (dict(ratio=-2), gp.CSA_ERR_INVALID_VALUE),
    # workspaces smaller than one row group's partials plus the status block
    (dict(ws=None), gp.CSA_ERR_WORKSPACE),
    (dict(ws_bytes=0), gp.CSA_ERR_WORKSPACE),
    (dict(ws_bytes=4 * 16 * 4 + 15), gp.CSA_ERR_WORKSPACE),  # ratio 4 x C 16 fp32 + 16 - 1
])
def test_bwd_rejects(lib, over, code):
    assert bwd_status(lib, **over) == code


def test_workspace_query_rejects_bad_sizes(lib):
    assert gp.csa_compressor_bwd_workspace_bytes(1, 4, 3, 8, 8, 2) == 0
    assert gp.csa_compressor_bwd_workspace_bytes(1, 200, 2, 12, 8, 2) == 0  # generic, window > 256


def test_test_hooks_range(lib):
    for bad in (-1, 1, gp.CSA_TEST_MIN_WAIT_CYCLES - 1, 5_000_000_000):
        assert lib.csa_compressor_test_hooks(bad, -1) == gp.CSA_ERR_INVALID_VALUE
    assert lib.csa_compressor_test_hooks(gp.CSA_TEST_MIN_WAIT_CYCLES, 3) == gp.CSA_OK
    assert lib.csa_compressor_test_hooks(0, -1) == gp.CSA_OK  # back to the defaults


def test_map_blocks_rejects(lib):
    assert lib.csa_compressor_map_blocks(None, 1, 4, 8, 2, FAKE, None, None) == gp.CSA_ERR_INVALID_VALUE
    assert lib.csa_compressor_map_blocks(FAKE, 1, 0, 8, 2, FAKE, None, None) == gp.CSA_ERR_INVALID_VALUE
    assert lib.csa_compressor_map_blocks(FAKE, 1, 4, 8, 2, None, None, None) == gp.CSA_ERR_INVALID_VALUE


def test_kpool_total_host_helper(lib, oracle_lib):
    rng = np.random.default_rng(1)
    for _ in range(50):
        S = int(rng.integers(0, 9))
        cu = np.concatenate([[0], np.cumsum(rng.integers(0, 40, S))]).astype(np.int32)
        lead = rng.integers(0, 12, S).astype(np.int32) if rng.random() < 0.7 else None
        P = int(rng.integers(1, 9))
        assert gp.csa_kpool_total(cu, lead, S, P) == oracle.kpool_total(cu, lead, P)
    assert gp.csa_kpool_total(np.array([0, 5, 3], np.int32), None, 2, 2) == -1
    assert gp.csa_kpool_total(np.array([0, 5], np.int32), np.array([-1], np.int32), 1, 2) == -1
    assert gp.csa_kpool_total(np.array([0, 5], np.int32), None, 1, 0) == -1


def kpool_status(lib, **over):
    a = dict(key=FAKE, gate=FAKE, cu=FAKE, lead=None, S=1, pool=4, d=8, capacity=8, out=FAKE,
             out_rows=2, compress=0, err=None)
    a.update(over)
    return lib.csa_kpool_fwd(a["key"], a["gate"], a["cu"], a["lead"], a["S"], a["pool"], a["d"],
                             a["capacity"], a["out"], a["out_rows"], a["compress"], a["err"], None)


@pytest.mark.parametrize("over,code", [
    (dict(S=-1), gp.CSA_ERR_INVALID_VALUE),
    (dict(pool=0), gp.CSA_ERR_INVALID_VALUE),
    (dict(d=0), gp.CSA_ERR_INVALID_VALUE),
    (dict(capacity=-1), gp.CSA_ERR_INVALID_VALUE),
    (dict(out_rows=-1), gp.CSA_ERR_INVALID_VALUE),
    (dict(compress=2), gp.CSA_ERR_INVALID_VALUE),
    (dict(cu=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(key=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(gate=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(out=None), gp.CSA_ERR_INVALID_VALUE),
    (dict(key=FAKE + 1), gp.CSA_ERR_INVALID_VALUE),
    (dict(lead=FAKE + 2), gp.CSA_ERR_INVALID_VALUE),
    (dict(err=FAKE + 2), gp.CSA_ERR_INVALID_VALUE),
    (dict(S=20000), gp.CSA_ERR_UNSUPPORTED),
    (dict(pool=gp.CSA_KPOOL_MAX_POOL + 1), gp.CSA_ERR_UNSUPPORTED),
    (dict(capacity=1 << 28, d=64), gp.CSA_ERR_UNSUPPORTED),
    (dict(out_rows=1 << 28, d=64), gp.CSA_ERR_UNSUPPORTED),
    (dict(S=0), gp.CSA_OK),  # no segment: nothing to enqueue
])
def test_kpool_rejects(lib, over, code):
    assert kpool_status(lib, **over) == code

