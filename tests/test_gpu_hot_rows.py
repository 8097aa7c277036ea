"""Backward with hot rows.  The workspace keeps the rows most looked up by the
previous backward; their gradients come from the per-bag histogram times the
gradient rows instead of the sort.  A first call learns the set; a second
call on the same inputs (weights and momentum reset) must still match the
oracle, including per-sample weights, long and short cold runs, and hot rows
that the batch does not touch."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe

CASES = {
    "hot": dict(name="hot", B=2048, E_scale=0.01),
    "weighted": dict(name="weighted", B=1024, T=16, E_scale=0.01),
    "small": dict(name="small", B=8192),
    "mixed": dict(name="mixed", B=2048, E_scale=0.05),
}


def make(case, seed=0):
    kw = dict(CASES[case])
    return workloads.make(kw.pop("name"), seed=seed, **kw)


def check_step(run, w, flags=0):
    hw = H.host(w)
    W_gpu, m_gpu = run.backward(flags)
    W_ref, m_ref = oracle.backward_rowwise_adagrad(H.tables(w), w.B, hw["indices"], hw["offsets"],
                                                   hw["grad_out"], hw["weights"], hw["momentum"],
                                                   w.lr, w.eps, hw["psw"])
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)


@pytest.mark.parametrize("two_launch", [False, True])
@pytest.mark.parametrize("case", list(CASES))
def test_backward_with_learned_hot_rows(case, two_launch):
    w = make(case)
    run = H.Run(w)
    flags = tbe.TBE_F_LONG_TWO_LAUNCH if two_launch else 0
    check_step(run, w, flags)            # fresh workspace: no hot rows yet
    hot = run.hot_set()
    if case in ("hot", "weighted", "small"):
        assert sum(len(h) for h in hot) > 0
    run.reset_state()
    check_step(run, w, flags)            # now with the hot rows
    # the hot set is kept: a third call still matches
    run.reset_state()
    check_step(run, w, flags)


def test_hot_rows_absent_from_the_batch_stay_untouched():
    w = make("hot", seed=1)
    run = H.Run(w)
    run.backward()
    hot = run.hot_set()
    assert sum(len(h) for h in hot) > 0
    # next batch: every lookup of a hot row of table 0 is moved to row 0
    hb = np.concatenate([[0], np.cumsum(w.E)])
    idx = w.indices.clone()
    t0_end = int(w.offsets[w.B])
    hot0 = torch.as_tensor(hot[0] - hb[0])
    mask = torch.isin(idx[:t0_end], hot0)
    idx[:t0_end][mask] = 0
    w2 = workloads.from_arrays(w.E, w.D, w.B, idx, w.offsets, w.weights, w.grad_out,
                               momentum=w.momentum, lr=w.lr, eps=w.eps)
    run.w = w2
    run.indices = idx.cuda()
    run.reset_state()
    check_step(run, w2)
    W_gpu = run.weights.cpu().numpy()
    for k in hot[0]:
        if k == 0:
            continue
        r = int(k - hb[0])
        D = int(w.D[0])
        assert np.array_equal(W_gpu[r * D:(r + 1) * D].view(np.uint16),
                              w.weights[r * D:(r + 1) * D].numpy().view(np.uint16))


def test_hot_set_carries_over_between_batches_of_different_sizes():
    # the hot set lives at a workspace offset that does not depend on n: a
    # batch with fewer lookups after a larger one still finds (and validates)
    # it, and the result matches the oracle
    w_big = make("hot", seed=2)
    run = H.Run(w_big)
    run.backward()
    hot = run.hot_set()
    assert sum(len(h) for h in hot) > 0
    B = w_big.B
    off = w_big.offsets.clone()
    # second batch: every bag keeps only its first half
    half = (off[1:] - off[:-1]) // 2
    keep = torch.cat([torch.arange(int(off[i]), int(off[i]) + int(half[i]))
                      for i in range(len(half))])
    idx2 = w_big.indices[keep]
    off2 = torch.cat([torch.zeros(1, dtype=off.dtype), torch.cumsum(half, 0).to(off.dtype)])
    w2 = workloads.from_arrays(w_big.E, w_big.D, B, idx2, off2, w_big.weights, w_big.grad_out,
                               momentum=w_big.momentum, lr=w_big.lr, eps=w_big.eps)
    assert w2.n < w_big.n
    run.w = w2
    run.indices, run.offsets = idx2.cuda(), off2.cuda()
    run.reset_state()
    check_step(run, w2)
    assert run.hot_set()[0].size > 0
