"""The oracle's OpenMP form (the timed CPU baseline) against the oracle itself:
the same forward outputs, weights and accumulators, bit for bit, for every
weight type, index type, pooling and Adagrad form, with out-of-range rows and
lookups past the last bag."""
import numpy as np
import pytest
import torch

import oracle
import oracle.openmp as omp
import workloads

CASES = {
    "tiny": dict(name="tiny"),
    "mixed": dict(name="mixed", B=256, E_scale=0.002),
    "weighted": dict(name="weighted", B=128, T=8, E_scale=0.002),
    "hot": dict(name="hot", B=64, T=2, E_scale=0.0005),
}


def _problem(case, seed=0, wdt=torch.float16):
    kw = dict(CASES[case])
    w = workloads.make(kw.pop("name"), seed=seed, weights_dtype=wdt, **kw)
    idx = w.indices.numpy().copy()
    off = w.offsets.numpy()
    # a few rows out of range (skipped by both) and two lookups past the last bag
    rng = np.random.default_rng(seed)
    bad = rng.choice(len(idx), size=max(1, len(idx) // 200), replace=False)
    idx[bad] = np.where(bad % 2 == 0, -1, 10 ** 6 * int(w.E.max()) % (2 ** 31 - 1))
    idx = np.concatenate([idx, np.zeros(2, idx.dtype)])
    return w, oracle.Tables(w.E, w.D), idx, off


def _weights(w, kind):
    if kind == "bf16":
        return w.weights.view(torch.int16).numpy().view(np.uint16)
    if kind == "fp32":
        return w.weights.float().numpy()
    return w.weights.numpy()


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("mean", [False, True])
def test_forward_equals_the_oracle(case, mean):
    w, tab, idx, off = _problem(case)
    psw = None if w.psw is None else np.concatenate([w.psw.numpy(), np.ones(2, np.float32)])
    W = _weights(w, "fp16")
    a = oracle.forward(tab, w.B, W, idx, off, psw, mean=mean)
    b = omp.forward(tab, w.B, W, idx, off, psw, mean=mean)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("kind", ["fp16", "bf16", "fp32"])
@pytest.mark.parametrize("mean,elementwise", [(False, False), (True, False), (False, True)])
def test_backward_equals_the_oracle(case, kind, mean, elementwise):
    wdt = torch.bfloat16 if kind == "bf16" else torch.float16
    w, tab, idx, off = _problem(case, seed=1, wdt=wdt)
    psw = None if w.psw is None else np.concatenate([w.psw.numpy(), np.ones(2, np.float32)])
    W = _weights(w, kind)
    rng = np.random.default_rng(2)
    size = int(tab.w_offsets[-1]) if elementwise else int(tab.hash_base[-1])
    m0 = rng.uniform(0, 0.5, size).astype(np.float32)
    G = w.grad_out.numpy()
    flags = dict(mean=mean, elementwise=elementwise, bf16=kind == "bf16", fp32=kind == "fp32")
    Wa, ma = oracle.backward_rowwise_adagrad(tab, w.B, idx, off, G, W, m0, w.lr, w.eps, psw,
                                             **flags)
    Wb, mb = omp.backward_rowwise_adagrad(tab, w.B, idx, off, G, W, m0, w.lr, w.eps, psw,
                                          **flags)
    assert np.array_equal(np.asarray(Wa).view(np.uint8), np.asarray(Wb).view(np.uint8))
    assert np.array_equal(ma.view(np.uint32), mb.view(np.uint32))
    assert not np.array_equal(ma, m0)  # the step did update rows


def test_runs_on_several_threads_and_rejects_bad_offsets():
    assert omp.threads() >= 1
    w, tab, idx, off = _problem("tiny")
    bad = off.copy()
    bad[3], bad[4] = bad[4], bad[3] - 1  # not monotone
    with pytest.raises(ValueError):
        omp.forward(tab, w.B, w.weights.numpy(), idx, bad)
    with pytest.raises(ValueError):
        omp.backward_rowwise_adagrad(tab, w.B, idx, bad, w.grad_out.numpy(), w.weights.numpy(),
                                     np.zeros(int(w.E.sum()), np.float32), w.lr, w.eps)
