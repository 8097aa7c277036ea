"""fp32 weights ("Forward: keep a narrowly specialized path beside the
general one": fp32 weights accumulate in fp64).  The forward's compensated
two-float accumulation must match the oracle's double sum to within one fp32
rounding plus (n 2^-24)^2 of the sum of |terms| (below 1e-9 of it here,
far tighter than a plain fp32 sum could meet); the backward's fp32 weights
and momentum must lie within the bound derived from its fp32 arithmetic, in
the row-wise and element-wise forms, fused and two-launch long runs, with
and without per-sample weights and mean pooling, through the workspace and
the no-allocation entry points."""
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
    "mixed": dict(name="mixed", B=512, E_scale=0.01),
    "weighted": dict(name="weighted", B=256, T=16, E_scale=0.01),
    "hot": dict(name="hot", B=256, T=2, E_scale=1e-4),
}


def make(case, seed=0):
    kw = dict(CASES[case])
    return workloads.make(kw.pop("name"), seed=seed, weights_dtype=torch.float32, **kw)


def _n_max(w):
    off = w.offsets.numpy().astype(np.int64)
    return int(np.diff(off).max()) if len(off) > 1 else 0


@pytest.mark.parametrize("mean", [False, True])
@pytest.mark.parametrize("case", list(CASES))
def test_fp32_forward_matches_oracle(case, mean):
    w = make(case)
    hw = H.host(w)
    tab = H.tables(w)
    ref = oracle.forward(tab, w.B, hw["weights"], hw["indices"], hw["offsets"], hw["psw"],
                         mean=mean, fp32=True)
    terms = oracle.forward(tab, w.B, np.abs(hw["weights"]), hw["indices"], hw["offsets"],
                           None if hw["psw"] is None else np.abs(hw["psw"]), mean=mean,
                           fp32=True)
    run = H.Run(w, weights_dtype=torch.float32, mean=mean)
    mflag = tbe.TBE_F_MEAN if mean else 0
    worst = H.assert_f32_forward_close(run.forward(mflag), ref, terms, _n_max(w), mean)
    print(f"{case}: worst |err| / sum|terms| = {worst:.2e}")
    # the preprocessed flag pools fp32 weights from the indices all the same
    tbe.tbe_preprocess(run.desc, run.indices, run.offsets, run.psw, run.ws)
    H.assert_f32_forward_close(run.forward(tbe.TBE_F_PREPROCESSED | mflag), ref, terms,
                               _n_max(w), mean)


@pytest.mark.parametrize("elementwise", [False, True])
@pytest.mark.parametrize("case", list(CASES))
def test_fp32_backward_matches_oracle(case, elementwise):
    w = make(case, seed=1)
    if elementwise:
        rng = np.random.default_rng(3)
        m0 = rng.uniform(0.01, 1.0, int(w.weights.numel())).astype(np.float32)
        w.momentum = torch.from_numpy(m0)
    hw = H.host(w)
    tab = H.tables(w)
    for flags in (0, tbe.TBE_F_LONG_TWO_LAUNCH):
        run = H.Run(w, weights_dtype=torch.float32, elementwise=elementwise)
        W_ref, m_ref = oracle.backward_rowwise_adagrad(
            tab, w.B, hw["indices"], hw["offsets"], hw["grad_out"], hw["weights"],
            hw["momentum"], w.lr, w.eps, hw["psw"], fp32=True, elementwise=elementwise)
        W_gpu, m_gpu = run.backward(flags)
        assert run.status() == 0
        H.assert_f32_step_close(tab, w.B, hw["indices"], hw["offsets"], hw["grad_out"],
                                hw["psw"], False, w.lr, w.eps, hw["weights"], hw["momentum"],
                                W_gpu, m_gpu, W_ref, m_ref, elementwise)


def test_fp32_mean_backward_and_noalloc():
    w = make("weighted", seed=2)
    hw = H.host(w)
    tab = H.tables(w)
    W_ref, m_ref = oracle.backward_rowwise_adagrad(
        tab, w.B, hw["indices"], hw["offsets"], hw["grad_out"], hw["weights"], hw["momentum"],
        w.lr, w.eps, hw["psw"], mean=True, fp32=True)
    run = H.Run(w, weights_dtype=torch.float32, mean=True)
    W_gpu, m_gpu = run.backward(tbe.TBE_F_MEAN)
    H.assert_f32_step_close(tab, w.B, hw["indices"], hw["offsets"], hw["grad_out"], hw["psw"],
                            True, w.lr, w.eps, hw["weights"], hw["momentum"], W_gpu, m_gpu,
                            W_ref, m_ref)
    # the no-allocation entry point on the same problem
    run2 = H.Run(w, weights_dtype=torch.float32)
    tbe.tbe_backward_rowwise_adagrad_noalloc(run2.desc, run2.grad_out, run2.indices,
                                             run2.offsets, run2.psw, run2.weights,
                                             run2.momentum, w.lr, w.eps, tbe.TBE_F_MEAN)
    torch.cuda.synchronize()
    H.assert_f32_step_close(tab, w.B, hw["indices"], hw["offsets"], hw["grad_out"], hw["psw"],
                            True, w.lr, w.eps, hw["weights"], hw["momentum"],
                            run2.weights.cpu().numpy(), run2.momentum.cpu().numpy(), W_ref,
                            m_ref)


def test_fp32_module_trains_two_steps():
    """Two steps through the module class: the second starts from the first's
    fp32 weights and momentum, against the oracle run twice."""
    w = make("mixed", seed=4)
    hw = H.host(w)
    tab = H.tables(w)
    model = tbe.TableBatchedEmbedding(w.E, w.D, w.B, w.n, weights=w.weights.cuda().clone(),
                                      momentum=w.momentum.cuda().clone(), lr=w.lr, eps=w.eps,
                                      weights_dtype=torch.float32)
    idx, off, g = w.indices.cuda(), w.offsets.cuda(), w.grad_out.cuda()
    W, m = hw["weights"], hw["momentum"]
    for _ in range(2):
        W_prev, m_prev = W, m
        out = model.forward(idx, off).cpu().numpy()
        ref = oracle.forward(tab, w.B, W_prev, hw["indices"], hw["offsets"], fp32=True)
        terms = oracle.forward(tab, w.B, np.abs(W_prev), hw["indices"], hw["offsets"],
                               fp32=True)
        H.assert_f32_forward_close(out, ref, terms, _n_max(w))
        model.backward(g, idx, off)
        torch.cuda.synchronize()
        W, m = oracle.backward_rowwise_adagrad(tab, w.B, hw["indices"], hw["offsets"],
                                               hw["grad_out"], W_prev, m_prev, w.lr, w.eps,
                                               fp32=True)
        W_gpu, m_gpu = model.weights.cpu().numpy(), model.momentum.cpu().numpy()
        H.assert_f32_step_close(tab, w.B, hw["indices"], hw["offsets"], hw["grad_out"], None,
                                False, w.lr, w.eps, W_prev, m_prev, W_gpu, m_gpu, W, m)
        # the next step compares against the oracle from the GPU's state
        W, m = W_gpu, m_gpu
