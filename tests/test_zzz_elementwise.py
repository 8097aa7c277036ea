"""Element-wise Adagrad (TBE_F_ELEMENTWISE): the HugeCTR page's Adagrad
kernel, one fp32 accumulator per weight element laid out like the weights,
m_c += g_c^2 and w_c -= lr g_c / (sqrt(m_c) + eps), with the same runs, hot
rows and gradient sums as the row-wise update.  The CUDA path against the
oracle's element-wise mode: short, medium and long runs (both long-run
variants), hot rows (the second step of a hot workload), per-sample weights,
mean pooling, bf16 weights, the no-alloc entry point, and the alignment the
accumulator rows need.  Initial accumulators are seeded draws in [0.01, 1).
The bound: one accumulator's increment g^2 exposes the fp32 rounding of its
gradient sum directly (the row-wise form averages it over the row), so each
element is held to an error bound derived from its own terms (see
assert_elementwise_step_close), and nearly all to 1e-5 / 1 ulp."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe
EW = tbe.TBE_F_ELEMENTWISE

CASES = {
    "tiny": dict(name="tiny"),
    "hot": dict(name="hot", B=2048, E_scale=0.01),
    "weighted": dict(name="weighted", B=1024, T=16, E_scale=0.01),
    "mixed": dict(name="mixed", B=2048, E_scale=0.05),
}


def make(case, seed=0, weights_dtype=torch.float16):
    kw = dict(CASES[case])
    w = workloads.make(kw.pop("name"), seed=seed, weights_dtype=weights_dtype, **kw)
    g = torch.Generator().manual_seed(1000 + seed)
    nW = int((w.E * w.D).sum())
    m0 = 0.01 + 0.99 * torch.rand(nW, generator=g)
    return dataclasses.replace(w, momentum=m0)


def host_weights(w):
    if w.weights.dtype == torch.bfloat16:
        return H.bf16_bits(w.weights)
    return w.weights.numpy()


def oracle_backward(w, mean=False):
    t = lambda x: None if x is None else x.numpy()
    return oracle.backward_rowwise_adagrad(
        H.tables(w), w.B, t(w.indices), t(w.offsets), t(w.grad_out), host_weights(w),
        t(w.momentum), w.lr, w.eps, t(w.psw), mean=mean,
        bf16=w.weights.dtype == torch.bfloat16, elementwise=True)


def check(run, w, flags=0, mean=False, max_loose=1e-3):
    W_ref, m_ref = oracle_backward(w, mean)
    W_gpu, m_gpu = run.backward(flags)
    t = lambda x: None if x is None else x.numpy()
    H.assert_elementwise_step_close(
        H.tables(w), w.B, t(w.indices), t(w.offsets), t(w.grad_out), t(w.psw), mean, w.lr,
        w.eps, host_weights(w), t(w.momentum), W_gpu, m_gpu, W_ref, m_ref,
        bf16=w.weights.dtype == torch.bfloat16, max_loose=max_loose)
    m0 = w.momentum.numpy()
    assert (m_ref != m0).any() and not np.array_equal(m_gpu, m0)


@pytest.mark.parametrize("case", list(CASES))
def test_elementwise_backward_matches_oracle(case):
    w = make(case)
    run = H.Run(w, elementwise=True)
    check(run, w)


@pytest.mark.parametrize("two_launch", [False, True])
def test_elementwise_long_run_variants(two_launch):
    w = make("hot", seed=2)
    run = H.Run(w, elementwise=True)
    assert run.preprocess()["n_long"] > 0
    check(run, w, tbe.TBE_F_LONG_TWO_LAUNCH if two_launch else 0)


@pytest.mark.parametrize("case", ["hot", "weighted"])
def test_elementwise_hot_rows(case):
    # a first step learns the hot set; the second, from the same state, updates
    # the hot rows through the tensor-core gradient and the hot-row finisher
    w = make(case, seed=5)
    run = H.Run(w, elementwise=True)
    run.backward()
    assert sum(len(h) for h in run.hot_set()) > 0
    run.reset_state()
    tbe.tbe_preprocess(run.desc, run.indices, run.offsets, run.psw, run.ws)
    # the hot rows' tensor-core gradient is held to the same allowance as the
    # cold rows' fp32 sums: its accumulator is flushed into fp32 partials
    # every few stages, so the tensor core's own accumulation error stays
    # within that of an fp32 sum
    check(run, w, tbe.TBE_F_PREPROCESSED, max_loose=1e-3)


def test_elementwise_with_mean_pooling():
    w = make("weighted", seed=6)
    run = H.Run(w, mean=True, elementwise=True)
    check(run, w, tbe.TBE_F_MEAN, mean=True)


@pytest.mark.parametrize("case", ["tiny", "mixed"])
def test_elementwise_with_bf16_weights(case):
    w = make(case, seed=7, weights_dtype=torch.bfloat16)
    run = H.Run(w, weights_dtype=torch.bfloat16, elementwise=True)
    check(run, w)


def test_elementwise_noalloc():
    w = make("tiny", seed=8)
    run = H.Run(w)
    W_ref, m_ref = oracle_backward(w)
    tbe.tbe_backward_rowwise_adagrad_noalloc(run.desc, run.grad_out, run.indices, run.offsets,
                                             run.psw, run.weights, run.momentum, w.lr, w.eps,
                                             flags=EW)
    torch.cuda.synchronize()
    t = lambda x: None if x is None else x.numpy()
    H.assert_elementwise_step_close(
        H.tables(w), w.B, t(w.indices), t(w.offsets), t(w.grad_out), t(w.psw), False, w.lr,
        w.eps, host_weights(w), t(w.momentum), run.weights.cpu().numpy(),
        run.momentum.cpu().numpy(), W_ref, m_ref)


def test_elementwise_needs_16_byte_aligned_accumulators():
    w = make("tiny", seed=9)
    run = H.Run(w, elementwise=True)
    nW = run.desc.num_weights
    buf = torch.zeros(nW + 4, dtype=torch.float32, device="cuda")
    launches = tbe.tbe_kernel_launches()
    with pytest.raises(RuntimeError):
        tbe.tbe_backward_rowwise_adagrad(run.desc, run.grad_out, run.indices, run.offsets,
                                         run.psw, run.weights, buf[1:], w.lr, w.eps, run.ws, EW)
    assert tbe.tbe_kernel_launches() == launches
