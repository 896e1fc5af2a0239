"""The roofline numerator. bench.py counts the consumed (token, column) slots of a pack in
closed form (coff=2: d * ratio * (2n - 1) per segment with n >= 1 blocks; coff=1:
d * ratio * n); the oracle, independently, records how many window positions read each
slot. The two must agree, every consumed slot having exactly one reader, and the
headline pack's algorithmic bytes are the figures the measurements are quoted on."""
import numpy as np
import pytest

import bench
import oracle
import thd_synth as ts

PACKS = {
    "tiny": ts.make_pack("tiny"),
    "r4c2_ragged": ts.make_custom([37, 12, 3, 0, 9, 4], ratio=4, coff=2, d=8, pad_rows=3, seed=1),
    "r2c1": ts.make_custom([5, 8, 1, 16, 0], ratio=2, coff=1, d=16, pad_rows=2, seed=2),
    "r32c2": ts.make_custom([130, 64, 7, 31], ratio=32, coff=2, d=8, pad_rows=1, seed=3),
    "r1c2": ts.make_custom([3, 1, 2], ratio=1, coff=2, d=8, pad_rows=0, seed=4),
}


@pytest.mark.parametrize("name", sorted(PACKS))
def test_consumed_slots_match_oracle_owners(name):
    pack = PACKS[name]
    owners = oracle.bwd_pack(pack, want_owners=True)["owners"]
    assert owners.max() <= 1
    assert bench.consumed_slots(pack) == int(np.count_nonzero(owners))


def test_headline_algorithmic_bytes():
    fwd, bwd = bench.algorithmic_bytes(ts.make_pack("3x8192_d512"))
    # kv + score 100.6 MB, out 6.3 MB, ape 16 KB, cu_seqlens 16 B (forward); the backward
    # adds dout and the full dKV/dScore writes, and reads and writes dAPE
    assert (fwd, bwd) == (106946576, 207626256)
