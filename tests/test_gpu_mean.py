"""Mean pooling (TBE_F_MEAN): the HugeCTR page's mean combiner, a bag of
L > 1 lookups pooled to its sum times 1/L and its gradient row scaled by 1/L
before the regrouping.  The CUDA path against the oracle's mean mode on the
plain forward (the small-table path is not taken), the preprocessed forward
with and without hot rows, and the backward (short, medium and long runs,
hot rows, the no-alloc entry point), plus bags of 0 and 1 lookups and bags
with out-of-range lookups (which count in L)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe
MEAN = tbe.TBE_F_MEAN

CASES = {
    "tiny": dict(name="tiny"),
    "hot": dict(name="hot", B=2048, E_scale=0.01),
    "weighted": dict(name="weighted", B=1024, T=16, E_scale=0.01),
    "small": dict(name="small", B=4096),
    "mixed": dict(name="mixed", B=2048, E_scale=0.05),
}


def make(case, seed=0):
    kw = dict(CASES[case])
    return workloads.make(kw.pop("name"), seed=seed, **kw)


def oracle_forward(w):
    hw = H.host(w)
    tab = H.tables(w)
    ref = oracle.forward(tab, w.B, hw["weights"], hw["indices"], hw["offsets"], hw["psw"], mean=True)
    absp = None if hw["psw"] is None else np.abs(hw["psw"])
    terms = oracle.forward(tab, w.B, np.abs(hw["weights"]), hw["indices"], hw["offsets"], absp,
                           mean=True)
    return ref, terms


def oracle_backward(w):
    hw = H.host(w)
    return oracle.backward_rowwise_adagrad(H.tables(w), w.B, hw["indices"], hw["offsets"],
                                           hw["grad_out"], hw["weights"], hw["momentum"], w.lr,
                                           w.eps, hw["psw"], mean=True)


@pytest.mark.parametrize("case", list(CASES))
def test_mean_forward_matches_oracle(case):
    w = make(case)
    run = H.Run(w, mean=True)
    ref, terms = oracle_forward(w)
    H.assert_forward_close(run.forward(MEAN), ref, terms)


@pytest.mark.parametrize("case", ["hot", "weighted", "mixed"])
def test_mean_preprocessed_forward_and_backward_match_oracle(case):
    w = make(case)
    run = H.Run(w, mean=True)
    ref, terms = oracle_forward(w)
    W_ref, m_ref = oracle_backward(w)
    # no hot set yet: cold lists only, then a backward learns one
    tbe.tbe_preprocess(run.desc, run.indices, run.offsets, run.psw, run.ws)
    H.assert_forward_close(run.forward(tbe.TBE_F_PREPROCESSED | MEAN), ref, terms)
    W1, m1 = run.backward(tbe.TBE_F_PREPROCESSED | MEAN)
    H.assert_momentum_close(m1, m_ref)
    H.assert_weights_within_ulp(W1, W_ref)
    run.reset_state()
    if case in ("hot", "weighted"):
        assert sum(len(h) for h in run.hot_set()) > 0
    # with hot rows (tensor-core forward and gradient)
    tbe.tbe_preprocess(run.desc, run.indices, run.offsets, run.psw, run.ws)
    H.assert_forward_close(run.forward(tbe.TBE_F_PREPROCESSED | MEAN), ref, terms)
    W2, m2 = run.backward(tbe.TBE_F_PREPROCESSED | MEAN)
    H.assert_momentum_close(m2, m_ref)
    H.assert_weights_within_ulp(W2, W_ref)


@pytest.mark.parametrize("two_launch", [False, True])
def test_mean_backward_without_preprocess_flag(two_launch):
    w = make("mixed", seed=3)
    run = H.Run(w, mean=True)
    W_ref, m_ref = oracle_backward(w)
    W_gpu, m_gpu = run.backward(MEAN | (tbe.TBE_F_LONG_TWO_LAUNCH if two_launch else 0))
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)


def test_mean_edge_bags():
    # bags of 0 and 1 lookups (unscaled), identical rows (the mean is the
    # row), and bags with out-of-range rows (they count in L)
    rng = np.random.default_rng(5)
    E, D, B = [40, 30], [16, 64], 8
    bags = [[[], [3], [7] * 9, [1, 45, -2, 2], list(rng.integers(0, 40, 200)), [0, 0],
             [39] * 129, list(rng.integers(0, 40, 17))],
            [[29], [], [5, 5, 5], list(rng.integers(0, 30, 70)), [31], [1, 2, 3, 4],
             [0] * 300, [10]]]
    idx, off = [], [0]
    for t in range(2):
        for b in range(B):
            idx.extend(bags[t][b])
            off.append(len(idx))
    W = (rng.standard_normal(int(np.dot(E, D))) * 0.01).astype(np.float16)
    G = rng.standard_normal((B, sum(D))).astype(np.float32)
    w = workloads.from_arrays(E, D, B, np.asarray(idx, np.int64), np.asarray(off, np.int64), W, G)
    run = H.Run(w, mean=True)
    ref, terms = oracle_forward(w)
    H.assert_forward_close(run.forward(MEAN), ref, terms)
    W_ref, m_ref = oracle_backward(w)
    W_gpu, m_gpu = run.backward(MEAN)
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)


def test_mean_noalloc_matches_oracle():
    w = make("tiny", seed=1)
    run = H.Run(w, mean=True)
    W_ref, m_ref = oracle_backward(w)
    tbe.tbe_backward_rowwise_adagrad_noalloc(run.desc, run.grad_out, run.indices, run.offsets,
                                             run.psw, run.weights, run.momentum, w.lr, w.eps,
                                             flags=MEAN)
    torch.cuda.synchronize()
    H.assert_momentum_close(run.momentum.cpu().numpy(), m_ref)
    H.assert_weights_within_ulp(run.weights.cpu().numpy(), W_ref)


def test_mean_backward_needs_a_mean_workspace():
    w = make("tiny")
    run = H.Run(w)  # workspace without TBE_WS_MEAN
    with pytest.raises(RuntimeError):
        run.backward(MEAN)
