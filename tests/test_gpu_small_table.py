"""The small-table forward (histogram counts times the table on the tensor
cores) against the oracle: ragged last tiles, every eligible width class,
tables shorter than 64 rows, counts above 2047 (exact only with the split
count operand) and out-of-range rows."""
import numpy as np
import pytest

import oracle
import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe


def small_problem(E, D, B, L, seed=0, repeat=None):
    rng = np.random.default_rng(seed)
    bags = [list(rng.integers(0, E, L)) for _ in range(B)]
    if repeat is not None:
        bags[B // 2] = [repeat[0]] * repeat[1] + bags[B // 2]
    idx = np.array([r for bg in bags for r in bg], np.int64)
    off = np.concatenate([[0], np.cumsum([len(b) for b in bags])]).astype(np.int64)
    W = rng.normal(0, 0.01, E * D).astype(np.float16)
    G = rng.normal(0, 1, (B, D)).astype(np.float32)
    return workloads.from_arrays([E], [D], B, idx, off, W, G)


def check_forward(w, flags=0):
    hw = H.host(w)
    run = H.Run(w)
    tab = H.tables(w)
    ref = oracle.forward(tab, w.B, hw["weights"], hw["indices"], hw["offsets"])
    terms = oracle.forward(tab, w.B, np.abs(hw["weights"]), hw["indices"], hw["offsets"])
    H.assert_forward_close(run.forward(flags), ref, terms)
    H.assert_forward_close(run.forward(tbe.TBE_F_FORCE_GENERIC), ref, terms)
    return run


@pytest.mark.parametrize("E,D,B,L", [(64, 128, 300, 128), (10, 64, 130, 64), (64, 96, 129, 100),
                                     (33, 80, 1, 70), (64, 112, 1000, 96), (1, 128, 128, 64)])
def test_small_table_matches_oracle(E, D, B, L):
    check_forward(small_problem(E, D, B, L, seed=E + D))


def test_small_table_counts_beyond_fp16_integers():
    # one bag holds row 5 five thousand times: count 5000 needs the split operand
    check_forward(small_problem(64, 128, 256, 64, seed=3, repeat=(5, 5000)))


def test_small_table_out_of_range_rows():
    w = small_problem(64, 128, 200, 64, seed=4)
    w.indices[::17] = 70  # beyond E
    w.indices[5] = -2
    run = check_forward(w, tbe.TBE_F_CHECK_BOUNDS)
    assert run.status() == tbe.TBE_ERR_INDEX_RANGE
