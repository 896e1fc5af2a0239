"""Launch planning, checked on the host (no GPU): tests/plan_check.cu is linked against the
library's objects and sweeps ratios, coff, head dims, segment and row counts. It checks
that every long-window, block-streaming and register-load plan fits the shared-memory
limit and the layout its kernel indexes (slices covering d, a stage per consumer group,
swizzle-aligned stages, tensor boxes of at most 256 rows, the ape area below the ring),
that every shape within the header's limits gets a plan and that plan a kernel, that the
slice-width rule picks 32 columns for few rows or head dims off a multiple of 64, and that
the row-group count never leaves CTAs for a second wave."""
import os
import subprocess

import pytest

from gated_pooling_gb300 import build as gb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OBJECTS = ["csa_fwd.o", "csa_bwd.o", "csa_api.o", "csa_noalloc.o", "csa_kpool.o"]


def test_plans_fit_the_device_and_the_kernels(tmp_path):
    try:
        cc = gb.nvcc()
    except RuntimeError as e:
        pytest.skip(str(e))
    gb.build()  # the library's objects (a no-op when they are current)
    objs = [os.path.join(gb.LIBDIR, o) for o in OBJECTS]
    for o in objs:
        assert os.path.exists(o), o
    exe = str(tmp_path / "plan_check")
    res = subprocess.run(
        [cc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
         "-I", os.path.join(ROOT, "gated_pooling_gb300", "csrc"),
         os.path.join(ROOT, "tests", "plan_check.cu")] + objs + ["-o", exe],
        capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    run = subprocess.run([exe], capture_output=True, text=True)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.startswith("ok "), run.stdout
