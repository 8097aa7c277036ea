"""Two independent problems, each with its own workspace, driven from two
streams at once: every call of one problem is enqueued between calls of the
other, so their kernels (and the side streams the library keeps per
workspace for the sort chain and the hot-row gradient) overlap on the GPU.
Each problem's forward and backward must match the oracle exactly as when it
runs alone (forward 1e-5 of the sum of |terms|, momentum 1e-5 relative,
weights 1 fp16 ulp)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe


def _expected(w):
    hw = H.host(w)
    tab = H.tables(w)
    ref = oracle.forward(tab, w.B, hw["weights"], hw["indices"], hw["offsets"], hw["psw"])
    terms = oracle.forward(tab, w.B, np.abs(hw["weights"]), hw["indices"], hw["offsets"],
                           None if hw["psw"] is None else np.abs(hw["psw"]))
    W, m = oracle.backward_rowwise_adagrad(tab, w.B, hw["indices"], hw["offsets"],
                                           hw["grad_out"], hw["weights"], hw["momentum"], w.lr,
                                           w.eps, hw["psw"])
    return ref, terms, W, m


@pytest.mark.parametrize("rounds", [3])
def test_two_workspaces_on_two_streams(rounds):
    wa = workloads.make("hot", seed=3, B=1024, T=4, E_scale=1e-3)       # byte tiles
    wb = workloads.make("weighted", seed=4, B=2048, T=8, E_scale=0.01)  # wide tiles
    runs = [H.Run(wa), H.Run(wb)]
    exp = [_expected(wa), _expected(wb)]
    for r in runs:  # hot sets from one serial step each
        r.backward()
        r.reset_state()
        assert sum(len(h) for h in r.hot_set()) > 0
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(rounds):
        for r in runs:
            r.reset_state()
        torch.cuda.synchronize()
        # preprocess, forward, backward of both problems, interleaved
        for i, r in enumerate(runs):
            with torch.cuda.stream(streams[i]):
                tbe.tbe_preprocess(r.desc, r.indices, r.offsets, r.psw, r.ws)
        for i, r in enumerate(runs):
            with torch.cuda.stream(streams[i]):
                tbe.tbe_forward(r.desc, r.weights, r.indices, r.offsets, r.psw, r.out, r.ws,
                                tbe.TBE_F_PREPROCESSED)
        for i, r in enumerate(runs):
            with torch.cuda.stream(streams[i]):
                tbe.tbe_backward_rowwise_adagrad(r.desc, r.grad_out, r.indices, r.offsets, r.psw,
                                                 r.weights, r.momentum, r.w.lr, r.w.eps, r.ws,
                                                 tbe.TBE_F_PREPROCESSED)
        torch.cuda.synchronize()
        for r, (ref, terms, W, m) in zip(runs, exp):
            assert r.status() == 0
            H.assert_forward_close(r.out.cpu().numpy(), ref, terms)
            H.assert_momentum_close(r.momentum.cpu().numpy(), m)
            H.assert_weights_within_ulp(r.weights.cpu().numpy(), W)
