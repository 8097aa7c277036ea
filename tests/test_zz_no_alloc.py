"""tbe_backward_rowwise_adagrad_noalloc: the backward for callers that must
not allocate device memory when they call it (serving engines and training
loops that hand out all device memory from their own pools up front, or that
cannot afford the device-wide synchronisation cudaMalloc/cudaFree may cause).
Its scratch is a fixed array inside the library.  Checked here against the
workspace entry point on the same inputs, two calls in a row, within the
tolerances of the other parity tests; and its size limit is checked."""
import numpy as np
import pytest
import torch

import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe


def _pair(w):
    """Two GPU copies of the same problem: one per entry point."""
    return H.Run(w), H.Run(w)


@pytest.mark.parametrize("recipe,kw", [("tiny", {}),
                                       ("weighted", dict(B=64, T=16, E_scale=0.01)),
                                       ("hot", dict(B=256, T=2, E_scale=0.01))])
@pytest.mark.parametrize("flags", [0, tbe.TBE_F_LONG_TWO_LAUNCH])
def test_noalloc_matches_workspace_entry_point_twice(recipe, kw, flags):
    w = workloads.make(recipe, seed=7, **kw)
    ref, got = _pair(w)
    for _ in range(2):  # the second call starts from the scratch the first one left
        # Each no-allocation call stands alone (no hot rows carried over), so
        # the workspace entry point gets a fresh workspace for each call too.
        ref.ws = tbe.Workspace(ref.desc, max(w.n, 1), w.psw is not None)
        tbe.tbe_backward_rowwise_adagrad(ref.desc, ref.grad_out, ref.indices, ref.offsets, ref.psw,
                                         ref.weights, ref.momentum, w.lr, w.eps, ref.ws, flags)
        tbe.tbe_backward_rowwise_adagrad_noalloc(got.desc, got.grad_out, got.indices, got.offsets,
                                                 got.psw, got.weights, got.momentum, w.lr, w.eps,
                                                 flags)
        torch.cuda.synchronize()
        H.assert_momentum_close(got.momentum.cpu().numpy(), ref.momentum.cpu().numpy())
        H.assert_weights_within_ulp(got.weights.cpu().numpy(), ref.weights.cpu().numpy())


def test_noalloc_rejects_problems_beyond_its_scratch():
    n = 4_000_000  # far more scratch than TBE_NOALLOC_SCRATCH_BYTES
    E, D, B = [1000], [128], 1
    idx = torch.zeros(n, dtype=torch.int64)
    off = torch.tensor([0, n], dtype=torch.int64)
    w = workloads.from_arrays(E, D, B, idx, off, np.zeros(1000 * 128, np.float16),
                              np.zeros((1, 128), np.float32))
    run = H.Run(w)
    with pytest.raises(tbe.TBEError) as err:
        tbe.tbe_backward_rowwise_adagrad_noalloc(run.desc, run.grad_out, run.indices, run.offsets,
                                                 None, run.weights, run.momentum, w.lr, w.eps)
    assert err.value.code == tbe.TBE_ETOO_LARGE
