"""Whole training steps captured into a CUDA graph and replayed.

Every backward joins the workspace's side-stream work (sort chain, hot-set
refresh) into its stream before it returns, so a step -- tbe_preprocess,
tbe_forward(TBE_F_PREPROCESSED), tbe_backward_rowwise_adagrad(TBE_F_PREPROCESSED)
-- can be captured, again and again on one workspace.  Replaying the graphs
must give bit for bit what the same steps give when launched one by one from
the same state (weights, momentum, workspace with its hot set): the kernels
sum in a fixed order whichever warp takes which task.  A step launched after
a replay, on the same workspace, continues from it.  The first replayed step
is also checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe

CASES = {
    "hot": dict(name="hot", B=4096, T=2, E_scale=1e-4),
    "mixed": dict(name="mixed", B=512, E_scale=0.01),
    "weighted": dict(name="weighted", B=256, T=16, E_scale=0.01),
}
PRE = tbe.TBE_F_PREPROCESSED


def _step(run):
    tbe.tbe_preprocess(run.desc, run.indices, run.offsets, run.psw, run.ws)
    tbe.tbe_forward(run.desc, run.weights, run.indices, run.offsets, run.psw, run.out, run.ws,
                    PRE)
    tbe.tbe_backward_rowwise_adagrad(run.desc, run.grad_out, run.indices, run.offsets, run.psw,
                                     run.weights, run.momentum, run.w.lr, run.w.eps, run.ws, PRE)


def _state(run):
    return (run.weights.clone(), run.momentum.clone(), run.ws.buf.clone())


def _restore(run, st):
    run.weights.copy_(st[0])
    run.momentum.copy_(st[1])
    run.ws.buf.copy_(st[2])


@pytest.mark.parametrize("case", list(CASES))
def test_graph_replay_matches_eager_steps(case):
    kw = dict(CASES[case])
    w = workloads.make(kw.pop("name"), seed=11, **kw)
    run = H.Run(w)
    for _ in range(2):  # learn a hot set, create the side stream
        _step(run)
    torch.cuda.synchronize()
    s0 = _state(run)
    hw = H.host(w)
    W0, m0 = run.host_weights(), run.momentum.cpu().numpy()

    # eager: two steps
    outs_e = []
    for _ in range(2):
        _step(run)
        outs_e.append(run.out.clone())
    torch.cuda.synchronize()
    W_e, m_e = run.weights.clone(), run.momentum.clone()

    # graphs: the same two steps from the same state, each captured into a
    # graph of its own on the same workspace (a later capture must not wait
    # on an earlier one's records), replayed in turn
    _restore(run, s0)
    torch.cuda.synchronize()
    graphs = [torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for g in graphs:
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                _step(run)
    torch.cuda.synchronize()
    _restore(run, s0)  # capture ran nothing, but start from the saved state all the same
    torch.cuda.synchronize()
    outs_g = []
    for g in graphs:
        g.replay()
        torch.cuda.synchronize()
        outs_g.append(run.out.clone())
    assert run.status() == 0
    for a, b in zip(outs_e, outs_g):
        assert torch.equal(a, b)
    assert torch.equal(run.weights.view(torch.int16), W_e.view(torch.int16))
    assert torch.equal(run.momentum, m_e)

    # and the first replayed step against the oracle
    tab = H.tables(w)
    W1, m1 = oracle.backward_rowwise_adagrad(tab, w.B, hw["indices"], hw["offsets"],
                                             hw["grad_out"], W0, m0, w.lr, w.eps, hw["psw"])
    _restore(run, s0)
    graphs[0].replay()
    torch.cuda.synchronize()
    ref = oracle.forward(tab, w.B, W0, hw["indices"], hw["offsets"], hw["psw"])
    terms = oracle.forward(tab, w.B, np.abs(W0), hw["indices"], hw["offsets"],
                           None if hw["psw"] is None else np.abs(hw["psw"]))
    H.assert_forward_close(run.out.cpu().numpy(), ref, terms)
    H.assert_momentum_close(run.momentum.cpu().numpy(), m1)
    H.assert_weights_within_ulp(run.host_weights(), W1)
    # a step launched after the replay continues from it: replayed first
    # step plus launched second step = the two launched steps
    _step(run)
    torch.cuda.synchronize()
    assert run.status() == 0
    assert torch.equal(run.out, outs_e[1])
    assert torch.equal(run.weights.view(torch.int16), W_e.view(torch.int16))
    assert torch.equal(run.momentum, m_e)
