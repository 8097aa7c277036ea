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


def _clamped_bags(off, n):
    """Each bag as the kernels read it without repair: [s, max(e, s)) with s
    and e clamped into [0, n] one by one (bags may overlap)."""
    o = np.clip(np.asarray(off, np.int64), 0, n)
    return [(int(o[i]), int(max(o[i + 1], o[i]))) for i in range(len(o) - 1)]


def test_malformed_offsets_without_repair_stay_in_bounds():
    """Offsets that are not monotone (overlapping bags whose lookups add up
    to far more than n), negative or beyond n, with no repair flag: every
    path (plain forward, preprocess, preprocessed forward with hot rows,
    backward, the no-allocation backward) must finish, report the bad
    offsets when asked, leave every row that no index names untouched, and
    leave the workspace fit for a well-formed batch afterwards.  The plain
    forward pools each bag over its own clamped range, which is checked
    against the oracle on rows gathered by numpy."""
    # E = 2000 rows per table: about 90 hot rows each, the rest of the lookups cold
    w = workloads.make("hot", B=256, E_scale=2e-4, T=2, seed=5)
    n = w.n
    good = w.offsets.numpy().copy()
    bad = good.copy()
    nb = len(bad) - 1
    bad[1:nb:2] = n          # bags 0, 2, 4, ...: [prev, n); bags 1, 3, ...: [n, 0) -> empty
    bad[2:nb:2] = 0
    bad[5], bad[9], bad[nb] = -7, n + 1000, n // 3
    wb = workloads.from_arrays(w.E, w.D, w.B, w.indices, bad, w.weights, w.grad_out,
                               momentum=w.momentum, lr=w.lr, eps=w.eps)
    run = H.Run(w)
    run.backward()  # a well-formed batch first: a hot set for the preprocessed paths
    run.reset_state()
    learned = run.hot_set()
    assert sum(len(h) for h in learned) > 0
    runb = H.Run(wb)
    runb.ws = run.ws  # same workspace, hot set included
    # plain forward: per-bag clamped ranges
    out = runb.forward(tbe.TBE_F_CHECK_BOUNDS)
    assert runb.status() == tbe.TBE_ERR_OFFSETS
    idx = w.indices.numpy().astype(np.int64)
    W = w.weights.numpy()
    W_off = np.concatenate([[0], np.cumsum(w.E * w.D)])
    D = int(w.D[0])
    for bag, (s, e) in enumerate(_clamped_bags(bad, n)):
        t, b = divmod(bag, w.B)
        rows = idx[s:e]
        rows = rows[(rows >= 0) & (rows < w.E[t])]
        g = W[W_off[t] + rows[:, None] * D + np.arange(D)[None, :]].reshape(len(rows), D)
        ref = oracle.pool_gathered([0, len(rows)], g)
        terms = oracle.pool_gathered([0, len(rows)], np.abs(g))
        # an fp32 sum of m terms is within (m - 1) 2^-24 of the sum of their
        # magnitudes: beyond 1e-5 for these bags of up to n lookups
        rel = max(1e-5, 1.1 * len(rows) * 2.0 ** -24)
        H.assert_forward_close(out[b:b + 1, t * D:(t + 1) * D], ref, terms, rel=rel)
    # preprocess + preprocessed forward + backward, and the plain backward
    named = np.zeros(int(w.E.sum()), bool)
    for t in range(w.T):
        r = idx[(idx >= 0) & (idx < w.E[t])]
        named[int(np.sum(w.E[:t])) + r] = True
    W0 = runb.host_weights().copy()
    m0 = runb.momentum.cpu().numpy().copy()
    pre = runb.preprocess(tbe.TBE_F_CHECK_BOUNDS)
    assert runb.status() == tbe.TBE_ERR_OFFSETS
    assert pre["n_valid"] <= n and pre["R"] <= n and pre["P"] <= n
    runb.forward(tbe.TBE_F_PREPROCESSED)
    for flags in (tbe.TBE_F_PREPROCESSED, 0, tbe.TBE_F_LONG_TWO_LAUNCH):
        W1, m1 = runb.backward(flags)
        assert runb.status() == 0
        assert np.isfinite(W1.astype(np.float32)).all() and np.isfinite(m1).all()
        rowmask = np.repeat(~named, D)
        assert np.array_equal(W1.view(np.uint16)[rowmask], W0.view(np.uint16)[rowmask])
        assert np.array_equal(m1.view(np.uint32)[~named], m0.view(np.uint32)[~named])
    tbe.tbe_backward_rowwise_adagrad_noalloc(runb.desc, runb.grad_out, runb.indices,
                                             runb.offsets, None, runb.weights, runb.momentum,
                                             w.lr, w.eps, 0)
    torch.cuda.synchronize()
    W1 = runb.host_weights()
    assert np.array_equal(W1.view(np.uint16)[np.repeat(~named, D)],
                          W0.view(np.uint16)[np.repeat(~named, D)])
    # the workspace still serves a well-formed batch exactly
    run.reset_state()
    hw = H.host(w)
    tab = H.tables(w)
    ref = oracle.forward(tab, w.B, hw["weights"], hw["indices"], hw["offsets"])
    terms = oracle.forward(tab, w.B, np.abs(hw["weights"]), hw["indices"], hw["offsets"])
    tbe.tbe_preprocess(run.desc, run.indices, run.offsets, None, run.ws)
    H.assert_forward_close(run.forward(tbe.TBE_F_PREPROCESSED), ref, terms)
    W_ref, m_ref = oracle.backward_rowwise_adagrad(tab, w.B, hw["indices"], hw["offsets"],
                                                   hw["grad_out"], hw["weights"], hw["momentum"],
                                                   w.lr, w.eps)
    W_gpu, m_gpu = run.backward(tbe.TBE_F_PREPROCESSED)
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)
