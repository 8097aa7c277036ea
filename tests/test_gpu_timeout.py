"""The bounded-wait time-out path of the tensor-core kernels, tested without
any fault or hang: a test-only build of the library (-DTBE_TEST_STUCK_WAIT)
makes the first ring wait of the hot forward's byte-tile kernel wait on an
mbarrier that nothing arrives on, bounded by a few thousand polls.  Every
CTA of that kernel then gives up, sets TBE_ERR_TIMEOUT in the workspace's
status word, drains the bulk copies it already issued under the normal bound
and frees its tensor memory.  The test reads the status bit through the C
ABI, and then checks that the context is still usable: a backward through
the same test build, and a forward through the regular build, match the
oracle."""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from table_embedding_bag_gb300 import _build
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe


@pytest.fixture(scope="module")
def stuck_lib(tmp_path_factory):
    d = tmp_path_factory.mktemp("stuck")
    path = _build.build(extra_flags=["-DTBE_TEST_STUCK_WAIT=4096"], lib=str(d / "libtbe_stuck.so"),
                        objdir=str(d / "obj"))
    assert os.path.exists(path)
    return tbe.configure(ctypes.CDLL(path))


def test_hot_forward_wait_times_out_and_reports(stuck_lib, monkeypatch):
    w = workloads.make("hot", seed=6, B=1024, T=2, E_scale=1e-3)
    run = H.Run(w)
    run.backward()  # regular build: learn a hot set, so the byte-tile kernel has tiles
    run.reset_state()
    assert sum(len(h) for h in run.hot_set()) > 0
    assert run.status() == 0
    hw = H.host(w)
    tab = H.tables(w)
    ref = oracle.forward(tab, w.B, hw["weights"], hw["indices"], hw["offsets"])
    terms = oracle.forward(tab, w.B, np.abs(hw["weights"]), hw["indices"], hw["offsets"])

    monkeypatch.setattr(tbe, "_lib", stuck_lib)
    tbe.tbe_preprocess(run.desc, run.indices, run.offsets, None, run.ws)
    run.out.fill_(0.0)
    tbe.tbe_forward(run.desc, run.weights, run.indices, run.offsets, None, run.out, run.ws,
                    tbe.TBE_F_PREPROCESSED)
    torch.cuda.synchronize()
    assert run.status() & tbe.TBE_ERR_TIMEOUT
    # the context still works: a backward through the test build (no stuck
    # wait on its path) matches the oracle
    W_ref, m_ref = oracle.backward_rowwise_adagrad(tab, w.B, hw["indices"], hw["offsets"],
                                                   hw["grad_out"], hw["weights"], hw["momentum"],
                                                   w.lr, w.eps)
    W_gpu, m_gpu = run.backward()
    assert run.status() == 0
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)
    monkeypatch.undo()
    # and the regular build's preprocessed forward is exact again
    run.reset_state()
    tbe.tbe_preprocess(run.desc, run.indices, run.offsets, None, run.ws)
    H.assert_forward_close(run.forward(tbe.TBE_F_PREPROCESSED), ref, terms)
    assert run.status() == 0
