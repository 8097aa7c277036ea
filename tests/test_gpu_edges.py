"""Edge cases of the CUDA path against the oracle: empty inputs, empty bags,
out-of-range rows, malformed offsets (checked and repaired), run lengths at
the short/long threshold, a run deep enough for a three-level reduction tree,
and the narrowest and widest table rows."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe


def custom(E, D, B, bags, seed=0, weighted=False, dtype=np.int64, lr=0.01, eps=1e-8):
    """bags: list (length T*B, table-major) of row lists."""
    rng = np.random.default_rng(seed)
    E, D = np.asarray(E), np.asarray(D)
    idx = np.array([r for bg in bags for r in bg], dtype=dtype)
    off = np.concatenate([[0], np.cumsum([len(b) for b in bags])]).astype(dtype)
    W = rng.normal(0, 0.01, int((E * D).sum())).astype(np.float16)
    G = rng.normal(0, 1, (B, int(D.sum()))).astype(np.float32)
    psw = rng.uniform(0, 1, len(idx)).astype(np.float32) if weighted else None
    m = rng.uniform(0, 0.1, int(E.sum())).astype(np.float32)
    return workloads.from_arrays(E, D, B, idx, off, W, G, psw=psw, momentum=m, lr=lr, eps=eps)


def check_all(w, flags=0, ulps=1):
    hw = H.host(w)
    run = H.Run(w)
    tab = H.tables(w)
    ref = oracle.forward(tab, w.B, hw["weights"], hw["indices"], hw["offsets"], hw["psw"])
    terms = oracle.forward(tab, w.B, np.abs(hw["weights"]), hw["indices"], hw["offsets"],
                           None if hw["psw"] is None else np.abs(hw["psw"]))
    H.assert_forward_close(run.forward(flags), ref, terms)
    W_ref, m_ref = oracle.backward_rowwise_adagrad(tab, w.B, hw["indices"], hw["offsets"],
                                                   hw["grad_out"], hw["weights"], hw["momentum"],
                                                   w.lr, w.eps, hw["psw"])
    W_gpu, m_gpu = run.backward(flags)
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref, ulps)
    return run


def test_no_lookups():
    w = custom([10, 20], [8, 16], 3, [[]] * 6)
    run = check_all(w)
    assert np.all(run.out.cpu().numpy() == 0)


def test_empty_bags_between_full_ones():
    bags = [[], [1, 2, 3], [], [], [0] * 40, []] + [[], [], [5], [], [], [2, 2]]
    check_all(custom([6, 7], [32, 64], 6, bags))


def test_single_table_single_bag():
    check_all(custom([5], [8], 1, [[0, 1, 2, 1, 4]]))


@pytest.mark.parametrize("D", [8, 24, 96, 160, 1024])
def test_row_widths(D):
    rng = np.random.default_rng(D)
    bags = [list(rng.integers(0, 50, rng.integers(0, 60))) for _ in range(16)]
    check_all(custom([50], [D], 16, bags, weighted=True))


@pytest.mark.parametrize("P", [1, 255, 256, 257, 511, 512, 513, 8191, 8192, 8193])
def test_run_lengths_around_chunk_boundaries(P):
    # row 3 is looked up by P distinct bags (a few of them twice); the work of
    # a run is counted in distinct bags, so P sits on the chunk boundaries
    rng = np.random.default_rng(P)
    B = P + 7
    bags = [[int(r)] for r in rng.integers(4, 10, B)]
    for b in range(P):
        bags[b] = [3] * (1 + (b % 5 == 0)) + bags[b]
    for flags in (0, tbe.TBE_F_LONG_TWO_LAUNCH):
        check_all(custom([10], [64], B, bags, seed=P, weighted=P % 2 == 1), flags)


def test_deep_reduction_tree():
    # one row looked up by 1.2M distinct bags: ~4700 chunks -> tree levels 147, 5, 1
    B = 1200000
    bags = [[7]] * B
    w = custom([9], [128], B, bags, seed=1)
    check_all(w)
    check_all(w, tbe.TBE_F_LONG_TWO_LAUNCH)


def test_out_of_range_rows_skipped_and_reported():
    bags = [[0, 1, -1, 2], [9, 3], [4, 100000, 4]] + [[1, -5], [2], [0, 0, 7]]
    w = custom([5, 3], [16, 8], 3, bags)
    hw = H.host(w)
    run = H.Run(w)
    tab = H.tables(w)
    ref = oracle.forward(tab, w.B, hw["weights"], hw["indices"], hw["offsets"])
    terms = oracle.forward(tab, w.B, np.abs(hw["weights"]), hw["indices"], hw["offsets"])
    H.assert_forward_close(run.forward(0), ref, terms)
    assert run.status() == 0  # checks off: skipped silently
    H.assert_forward_close(run.forward(tbe.TBE_F_CHECK_BOUNDS), ref, terms)
    assert run.status() == tbe.TBE_ERR_INDEX_RANGE
    W_ref, m_ref = oracle.backward_rowwise_adagrad(tab, w.B, hw["indices"], hw["offsets"],
                                                   hw["grad_out"], hw["weights"], hw["momentum"],
                                                   w.lr, w.eps)
    W_gpu, m_gpu = run.backward(tbe.TBE_F_CHECK_BOUNDS)
    assert run.status() == tbe.TBE_ERR_INDEX_RANGE
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)


def test_malformed_offsets_detected_and_repaired():
    w = custom([8, 8], [16, 16], 4, [[1, 2], [3], [], [4, 5, 6], [7], [0, 0], [1], [2, 3]])
    good = w.offsets.numpy().copy()
    n = len(w.indices)
    bad = good.copy()
    bad[2], bad[3], bad[5] = 9, 2, n + 4  # non-monotone and beyond n
    fixed, _ = oracle.repair_offsets(bad, n)
    wb = workloads.from_arrays(w.E, w.D, w.B, w.indices, bad, w.weights, w.grad_out,
                               momentum=w.momentum, lr=w.lr, eps=w.eps)
    wf = workloads.from_arrays(w.E, w.D, w.B, w.indices, fixed, w.weights, w.grad_out,
                               momentum=w.momentum, lr=w.lr, eps=w.eps)
    run = H.Run(wb)
    run.forward(tbe.TBE_F_CHECK_BOUNDS)
    assert run.status() == tbe.TBE_ERR_OFFSETS
    # repair mode: same results as the oracle on the repaired offsets
    hf = H.host(wf)
    tab = H.tables(wf)
    ref = oracle.forward(tab, wf.B, hf["weights"], hf["indices"], hf["offsets"])
    terms = oracle.forward(tab, wf.B, np.abs(hf["weights"]), hf["indices"], hf["offsets"])
    H.assert_forward_close(run.forward(tbe.TBE_F_REPAIR_OFFSETS), ref, terms)
    assert run.status() == tbe.TBE_ERR_OFFSETS
    W_ref, m_ref = oracle.backward_rowwise_adagrad(tab, wf.B, hf["indices"], hf["offsets"],
                                                   hf["grad_out"], hf["weights"], hf["momentum"],
                                                   wf.lr, wf.eps)
    W_gpu, m_gpu = run.backward(tbe.TBE_F_REPAIR_OFFSETS)
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)


def test_preprocessed_flag_reuses_runs():
    w = workloads.make("weighted", B=64, T=16, E_scale=0.01, seed=2)
    hw = H.host(w)
    run = H.Run(w)
    run.preprocess()
    W_gpu, m_gpu = run.backward(tbe.TBE_F_PREPROCESSED)
    W_ref, m_ref = oracle.backward_rowwise_adagrad(H.tables(w), w.B, hw["indices"], hw["offsets"],
                                                   hw["grad_out"], hw["weights"], hw["momentum"],
                                                   w.lr, w.eps, hw["psw"])
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)
