"""Forward from the preprocessed workspace (TBE_F_PREPROCESSED): each table's
hot rows through the tensor cores (per-bag histogram times the hot rows), the
cold lookups gathered from the per-bag cold lists.  That path is taken when
bags hold at least 64 lookups on average (hot, small and the custom cases
here); shorter bags (tiny, mixed, weighted recipes) are pooled from the
indices, which must give the same sums.  Compared with the
oracle's pooled sums before any hot set exists (cold lists only) and after a
backward has chosen one; edge cases cover counts past the tf32 significand,
per-sample weights of very different magnitudes, widths that are not a
multiple of the MMA's N step or too wide for hot rows, and empty batches."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe

CASES = {
    "tiny": dict(name="tiny"),
    "hot": dict(name="hot", B=2048, E_scale=0.01),
    "weighted": dict(name="weighted", B=1024, T=16, E_scale=0.01),
    "small": dict(name="small", B=8192),
    "mixed": dict(name="mixed", B=2048, E_scale=0.05),
}


def make(case, seed=0):
    kw = dict(CASES[case])
    return workloads.make(kw.pop("name"), seed=seed, **kw)


def oracle_forward(w):
    hw = H.host(w)
    tab = H.tables(w)
    ref = oracle.forward(tab, w.B, hw["weights"], hw["indices"], hw["offsets"], hw["psw"])
    absp = None if hw["psw"] is None else np.abs(hw["psw"])
    terms = oracle.forward(tab, w.B, np.abs(hw["weights"]), hw["indices"], hw["offsets"], absp)
    return ref, terms


def forward_preprocessed(run):
    tbe.tbe_preprocess(run.desc, run.indices, run.offsets, run.psw, run.ws)
    return run.forward(flags=tbe.TBE_F_PREPROCESSED)


def learn_hot_set(run):
    run.backward()
    run.reset_state()
    return run.hot_set()


@pytest.mark.parametrize("case", list(CASES))
def test_preprocessed_forward_matches_oracle(case):
    w = make(case)
    run = H.Run(w)
    ref, terms = oracle_forward(w)
    H.assert_forward_close(forward_preprocessed(run), ref, terms)   # no hot rows yet
    hot = learn_hot_set(run)
    if case in ("hot", "weighted", "small"):
        assert sum(len(h) for h in hot) > 0
    H.assert_forward_close(forward_preprocessed(run), ref, terms)   # with hot rows
    H.assert_forward_close(forward_preprocessed(run), ref, terms)   # set kept


def _custom(E, D, bags, seed=0, psw=None):
    """Workload from explicit per-table bag lists: bags[t][b] = list of rows."""
    rng = np.random.default_rng(seed)
    T, B = len(E), len(bags[0])
    idx, off = [], [0]
    for t in range(T):
        for b in range(B):
            idx.extend(bags[t][b])
            off.append(len(idx))
    W = (rng.standard_normal(int(np.dot(E, D))) * 0.01).astype(np.float16)
    G = rng.standard_normal((B, int(np.sum(D)))).astype(np.float32)
    return workloads.from_arrays(E, D, B, np.asarray(idx, np.int64), np.asarray(off, np.int64),
                                 W, G, psw=psw)


def test_counts_beyond_the_tf32_significand():
    # row 7 appears 5003 times in bag 0: the histogram's remainder term is 3
    rng = np.random.default_rng(3)
    bags = [[[7] * 5003 + list(rng.integers(0, 100, 10)), [], [7] * 300 + [3] * 2049,
             list(rng.integers(0, 100, 50))]]
    w = _custom([100], [64], bags)
    run = H.Run(w)
    ref, terms = oracle_forward(w)
    hot = learn_hot_set(run)
    assert 7 in set(hot[0].tolist()) and 3 in set(hot[0].tolist())
    H.assert_forward_close(forward_preprocessed(run), ref, terms)


def test_widths_padding_and_tables_too_wide_for_hot_rows():
    # D = 8 (N padded to 16), 136 (not a multiple of 32), 256 (widest hot
    # table), 512 (no hot rows): half of every bag hits four rows
    rng = np.random.default_rng(5)
    E, D, B, L = [50, 700, 1000, 300], [8, 136, 256, 512], 300, 160
    bags = []
    for t in range(len(E)):
        tb = []
        for b in range(B):
            n = int(rng.integers(0, L))
            hot = rng.integers(0, 4, n // 2)
            cold = rng.integers(0, E[t], n - n // 2)
            tb.append(list(rng.permutation(np.concatenate([hot, cold]))))
        bags.append(tb)
    w = _custom(E, D, bags)
    run = H.Run(w)
    ref, terms = oracle_forward(w)
    hot = learn_hot_set(run)
    assert all(len(hot[t]) > 0 for t in range(3)) and len(hot[3]) == 0
    H.assert_forward_close(forward_preprocessed(run), ref, terms)


def test_weighted_with_widely_spread_weights():
    rng = np.random.default_rng(9)
    E, D, B = [40, 5000], [32, 128], 256
    bags = [[list(rng.integers(0, 8, int(rng.integers(64, 192)))) for _ in range(B)]
            for _ in range(2)]
    n = sum(len(b) for t in bags for b in t)
    psw = (10.0 ** rng.uniform(-6, 3, n) * rng.choice([-1, 1], n)).astype(np.float32)
    w = _custom(E, D, bags, psw=psw)
    run = H.Run(w)
    ref, terms = oracle_forward(w)
    hot = learn_hot_set(run)
    assert all(len(h) > 0 for h in hot)
    H.assert_forward_close(forward_preprocessed(run), ref, terms)


def test_empty_batch_after_hot_rows_were_learned():
    w = make("hot")
    run = H.Run(w)
    assert sum(len(h) for h in learn_hot_set(run)) > 0
    run.indices = run.indices[:0]
    run.offsets = torch.zeros_like(run.offsets)
    run.psw = None
    out = forward_preprocessed(run)
    assert not out.any()


def test_counts_far_beyond_the_fp16_range():
    # counts of 40001 and 70000 lookups of one row in a bag: the forward's
    # scaled three-part fp16 split and the gradient's tf32 remainder terms
    # must keep forward and backward on the oracle
    rng = np.random.default_rng(11)
    bags = [[[7] * 40001 + [3] * 9, [7] * 5 + [3] * 70000, list(rng.integers(0, 50, 100)),
             [5] * 2048]]
    w = _custom([50], [64], bags)
    run = H.Run(w)
    ref, terms = oracle_forward(w)
    hot = learn_hot_set(run)
    assert {3, 5, 7} <= set(hot[0].tolist())
    H.assert_forward_close(forward_preprocessed(run), ref, terms)
    hw = H.host(w)
    W_gpu, m_gpu = run.backward(tbe.TBE_F_PREPROCESSED)
    W_ref, m_ref = oracle.backward_rowwise_adagrad(H.tables(w), w.B, hw["indices"], hw["offsets"],
                                                   hw["grad_out"], hw["weights"], hw["momentum"],
                                                   w.lr, w.eps, hw["psw"])
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)


def test_byte_and_wide_tiles_in_one_table():
    # 400 bags = three 128-bag tiles and a ragged one of 16.  Table 0: bag
    # 150 (second tile) and bag 390 (last tile) hold 300 lookups of one row,
    # past a byte, so those tiles keep fp32 rows; the others are byte tiles.
    # Table 1 stays in bytes (at most 255 of a row per bag, 255 in bag 7).
    rng = np.random.default_rng(13)
    E, D, B = [60, 3000], [64, 128], 400
    bags = []
    for t in range(2):
        tb = []
        for b in range(B):
            n = int(rng.integers(60, 140))
            hot = rng.integers(0, 6, n * 3 // 4)
            cold = rng.integers(0, E[t], n - n * 3 // 4)
            tb.append(list(rng.permutation(np.concatenate([hot, cold]))))
        bags.append(tb)
    bags[0][150] = bags[0][150] + [5] * 300
    bags[0][390] = [2] * 300 + bags[0][390]
    bags[1][7] = [4] * 255 + bags[1][7]
    w = _custom(E, D, bags)
    run = H.Run(w)
    ref, terms = oracle_forward(w)
    hot = learn_hot_set(run)
    assert all(len(h) > 0 for h in hot)
    H.assert_forward_close(forward_preprocessed(run), ref, terms)
    hw = H.host(w)
    W_gpu, m_gpu = run.backward(tbe.TBE_F_PREPROCESSED)
    W_ref, m_ref = oracle.backward_rowwise_adagrad(H.tables(w), w.B, hw["indices"], hw["offsets"],
                                                   hw["grad_out"], hw["weights"], hw["momentum"],
                                                   w.lr, w.eps, hw["psw"])
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)


def test_hot_sets_at_capacity_with_a_cold_remainder():
    # 300 and 310 rows, each looked up far above the hot threshold: the hot
    # sets are (nearly) full and the remaining rows stay cold.  Bag 200 of
    # table 0 has 300 lookups of one row (its tile keeps fp32 rows); table 1
    # (D = 256) stays in bytes.
    rng = np.random.default_rng(17)
    E, D, B = [300, 310], [64, 256], 384
    bags = [[list(rng.integers(0, E[t], int(rng.integers(80, 160)))) for _ in range(B)]
            for t in range(2)]
    bags[0][200] = bags[0][200] + [290] * 300
    w = _custom(E, D, bags)
    run = H.Run(w)
    ref, terms = oracle_forward(w)
    hot = learn_hot_set(run)
    slots = tbe.tbe_workspace_view(run.desc, max(w.n, 1), run.ws)["hot_slots"]
    # the selection cuts at log-scale count buckets, so a set of evenly used
    # rows need not fill every slot
    assert all(0 < len(h) <= min(slots, e) for h, e in zip(hot, E))
    H.assert_forward_close(forward_preprocessed(run), ref, terms)
    hw = H.host(w)
    W_gpu, m_gpu = run.backward(tbe.TBE_F_PREPROCESSED)
    W_ref, m_ref = oracle.backward_rowwise_adagrad(H.tables(w), w.B, hw["indices"], hw["offsets"],
                                                   hw["grad_out"], hw["weights"], hw["momentum"],
                                                   w.lr, w.eps, hw["psw"])
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)
