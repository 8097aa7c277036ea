"""Full-size workloads (the five recipes at their stated sizes, drawn on the
device, the launch configuration bench.py times) against the oracle on
sampled outputs, plus properties of the sort that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe

NAMES = ["small", "mixed", "weighted", "hot"]


@pytest.fixture(scope="module", params=NAMES)
def full(request):
    torch.cuda.empty_cache()
    w = workloads.make(request.param, device="cuda", seed=0)
    yield w
    del w
    torch.cuda.empty_cache()


def _host_inputs(w):
    return (w.indices.cpu().numpy(), w.offsets.cpu().numpy(),
            None if w.psw is None else w.psw.cpu().numpy())


def test_fullsize_forward_sampled_bags(full):
    w = full
    run = H.Run(w)
    run.weights = w.weights  # resident; forward does not modify it
    out = run.forward()
    idx, off, psw = _host_inputs(w)
    rng = np.random.default_rng(1)
    nb = w.T * w.B
    bags = np.unique(np.concatenate([[0, nb - 1], rng.integers(0, nb, 300)]))
    D_off = np.concatenate([[0], np.cumsum(w.D)])
    W_off = np.concatenate([[0], np.cumsum(w.E * w.D)])
    for t in np.unique(bags // w.B):
        tb = bags[bags // w.B == t]
        D = int(w.D[t])
        seg = [np.arange(off[b], off[b + 1]) for b in tb]
        pos = np.concatenate(seg) if seg else np.zeros(0, np.int64)
        rows = idx[pos].astype(np.int64)
        flat = torch.as_tensor(W_off[t] + rows[:, None] * D + np.arange(D)[None, :],
                               device="cuda")
        gathered = w.weights[flat.reshape(-1)].reshape(len(rows), D).cpu().numpy()
        bo = np.concatenate([[0], np.cumsum([len(s) for s in seg])])
        coef = None if psw is None else psw[pos]
        ref = oracle.pool_gathered(bo, gathered, coef)
        terms = oracle.pool_gathered(bo, np.abs(gathered), None if coef is None else np.abs(coef))
        got = out[tb % w.B, D_off[t]:D_off[t] + D]
        H.assert_forward_close(got, ref, terms)


def test_fullsize_sort_properties(full):
    w = full
    run = H.Run(w)
    got = run.preprocess()
    n = w.n
    assert got["n_valid"] == n  # every lookup of these recipes is in range
    keys = torch.from_numpy(got["sorted_keys"].view(np.int32)).long() & 0xffffffff
    bags = torch.from_numpy(got["sorted_bags"].view(np.int32)).long()
    # expected: every (key, bag) pair of the input, in (key, bag) order; a
    # stable sort of table-major lookups yields exactly that order
    t_of = torch.repeat_interleave(torch.arange(w.T * w.B, device="cuda") // w.B,
                                   (w.offsets[1:] - w.offsets[:-1]).long())
    b_of = torch.repeat_interleave(torch.arange(w.T * w.B, device="cuda") % w.B,
                                   (w.offsets[1:] - w.offsets[:-1]).long())
    hb = torch.as_tensor(np.concatenate([[0], np.cumsum(w.E)]), device="cuda")
    lin = hb[t_of] + w.indices.long()
    exp = torch.sort(lin * (1 << 32) + b_of).values.cpu()
    assert torch.equal(keys * (1 << 32) + bags, exp)
    # runs: starts strictly increase, first keys strictly increase and match
    rs = got["run_starts"].astype(np.int64)
    uk = got["unique_keys"].astype(np.int64)
    k = keys.numpy()
    assert rs[0] == 0 and rs[-1] == n and np.all(np.diff(rs) > 0)
    assert np.all(np.diff(uk) > 0) and np.array_equal(k[rs[:-1]], uk)
    assert got["R"] == int(np.count_nonzero(np.diff(k))) + 1
    ps, pb, rp = H.pair_structure(k, bags.numpy(), rs)
    assert got["P"] == len(pb)
    assert np.array_equal(got["pair_starts"].astype(np.int64), ps)
    assert np.array_equal(got["run_pairs"].astype(np.int64), rp)
    npairs = np.diff(rp)
    assert np.array_equal(np.sort(got["long_runs"]),
                          np.nonzero(npairs >= got["long_threshold"])[0])


@pytest.mark.parametrize("two_launch", [False, True])
def test_fullsize_backward_sampled_rows(full, two_launch):
    w = full
    run = H.Run(w)
    pre = run.preprocess()
    rp = pre["run_pairs"].astype(np.int64)
    uk = pre["unique_keys"].astype(np.int64)
    sl = np.diff(rp)
    rng = np.random.default_rng(2)
    # the longest runs (deepest reduction trees), random touched rows, and a
    # few untouched rows
    longest = uk[np.argsort(-sl)[:6]]
    touched = uk[rng.integers(0, len(uk), 200)]
    mask = np.ones(int(w.E.sum()), bool)
    mask[uk] = False
    free = np.nonzero(mask)[0]
    untouched = free[rng.integers(0, len(free), 20)] if len(free) else np.zeros(0, np.int64)
    sel = np.unique(np.concatenate([longest, touched, untouched])).astype(np.uint32)
    hb = np.concatenate([[0], np.cumsum(w.E)])
    W_off = np.concatenate([[0], np.cumsum(w.E * w.D)])
    maxD = int(w.D.max())
    t_sel = np.searchsorted(hb, sel, side="right") - 1

    def rows_of(weights_dev):
        out = np.zeros((len(sel), maxD), np.float16)
        for j, (k, t) in enumerate(zip(sel, t_sel)):
            D = int(w.D[t])
            s = int(W_off[t] + (int(k) - hb[t]) * D)
            out[j, :D] = weights_dev[s:s + D].cpu().numpy()
        return out

    w0 = rows_of(run.weights)
    m0 = run.momentum[torch.as_tensor(sel.astype(np.int64), device="cuda")].cpu().numpy()
    flags = tbe.TBE_F_PREPROCESSED | (tbe.TBE_F_LONG_TWO_LAUNCH if two_launch else 0)
    run.backward(flags)
    w1 = rows_of(run.weights)
    m1 = run.momentum[torch.as_tensor(sel.astype(np.int64), device="cuda")].cpu().numpy()
    idx, off, psw = _host_inputs(w)
    ws, ms, cnt = oracle.backward_selected(H.tables(w), w.B, idx, off, w.grad_out.cpu().numpy(),
                                           w.lr, w.eps, sel, w0, m0, psw)
    H.assert_momentum_close(m1, ms)
    H.assert_weights_within_ulp(w1, ws)
    untouched_sel = cnt == 0
    assert np.array_equal(w1[untouched_sel].view(np.uint16), w0[untouched_sel].view(np.uint16))
    assert np.array_equal(m1[untouched_sel].view(np.uint32), m0[untouched_sel].view(np.uint32))
