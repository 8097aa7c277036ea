"""The path bench.py times, checked against the oracle at sizes where its
tensor-core kernels loop: tbe_preprocess -> tbe_forward(TBE_F_PREPROCESSED)
-> tbe_backward_rowwise_adagrad(TBE_F_PREPROCESSED), fused and two-launch,
with a hot set learned by an earlier backward on the same batch (weights and
momentum reset afterwards, so the checked step starts from the workload's
values).

Sizes: the hot-row recipe at B = 32768 (tables shrunk to 1e5 rows), which
gives 2048 byte-histogram tiles, about 13 per CTA of the persistent hot
forward kernel (its ring refill and both tensor-memory accumulators run) and
about 27 stages per hot-gradient partition; the full hot-row recipe (B =
131072, about 54 tiles per CTA, 108 stages per partition); and the full
weighted recipe (wide fp32 histogram tiles in the hot-row gradient).

Checked ("Backward: invert 'which rows did this sample use?'": every touched
row updated exactly once): 300 sampled bags of the forward against
oracle.pool_gathered; the hot rows, the longest cold runs, random cold rows
and untouched rows after the backward against oracle.backward_selected.
Tolerances: forward 1e-5 of the sum of |terms|, momentum 1e-5 relative,
weights 1 fp16 ulp, untouched rows bit-identical."""
import numpy as np
import pytest
import torch

import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
tbe = H.tbe

CASES = {
    "hot_b32768": dict(name="hot", B=32768, E_scale=0.01),
    "hot_full": dict(name="hot"),
    "weighted_full": dict(name="weighted"),
}


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    torch.cuda.empty_cache()
    kw = dict(CASES[request.param])
    w = workloads.make(kw.pop("name"), device="cuda", seed=0, **kw)
    run = H.Run(w)
    # learn the hot set on this batch, then start the checked steps afresh
    run.backward()
    run.reset_state()
    inputs = H.host_inputs(w)
    yield request.param, w, run, inputs
    del run, w
    torch.cuda.empty_cache()


def _cold_runs(run):
    """Keys and pair counts of the cold runs of the last preprocess."""
    v = tbe.tbe_workspace_view(run.desc, run.w.n, run.ws)
    counts = H.ws_array(run.ws, v["counts"], 8)
    R = int(counts[0])
    uk = H.ws_array(run.ws, v["unique_keys"], R).astype(np.int64)
    rp = H.ws_array(run.ws, v["run_pairs"], R + 1).astype(np.int64)
    return uk, np.diff(rp), int(counts[1])


def _selection(w, hot, uk, sl, name):
    rng = np.random.default_rng(2)
    if name == "hot_full":
        # every hot row of table 0 and the two most looked-up of the others
        hot_sel = np.concatenate([hot[0]] + [h[:2] for h in hot[1:]]) if hot else []
    else:
        hot_sel = np.concatenate(hot) if hot else []
    longest = uk[np.argsort(-sl)[:6]]
    touched = uk[rng.integers(0, len(uk), 200)] if len(uk) else np.zeros(0, np.int64)
    mask = np.ones(int(w.E.sum()), bool)
    mask[uk] = False
    for h in hot:
        mask[h] = False
    free = np.nonzero(mask)[0]
    untouched = free[rng.integers(0, len(free), 20)] if len(free) else np.zeros(0, np.int64)
    sel = np.unique(np.concatenate([np.asarray(hot_sel, np.int64), longest, touched,
                                    untouched])).astype(np.uint32)
    return sel, len(hot_sel)


@pytest.mark.parametrize("two_launch", [False, True])
def test_benchmarked_step_with_learned_hot_set(case, two_launch):
    name, w, run, inputs = case
    run.reset_state()
    hot = run.hot_set()  # the set the preprocess below takes
    n_hot = sum(len(h) for h in hot)
    if name.startswith("hot"):
        assert n_hot >= 200 * w.T, n_hot  # the set holds nearly all of each table's 256 slots
    else:
        assert n_hot > 0

    tbe.tbe_preprocess(run.desc, run.indices, run.offsets, run.psw, run.ws)
    out = run.forward(flags=tbe.TBE_F_PREPROCESSED)
    assert H.check_sampled_bags(w, run.weights, out, nsample=300, inputs=inputs) >= 250

    uk, sl, n_cold = _cold_runs(run)
    sel, nh_sel = _selection(w, [h.astype(np.int64) for h in hot], uk, sl, name)
    w0, m0 = H.selected_rows(w, run.weights, run.momentum, sel)
    flags = tbe.TBE_F_PREPROCESSED | (tbe.TBE_F_LONG_TWO_LAUNCH if two_launch else 0)
    run.backward(flags)
    assert run.status() == 0
    w1, m1 = H.selected_rows(w, run.weights, run.momentum, sel)
    cnt = H.check_selected_rows(w, sel, w0, m0, w1, m1, inputs=inputs)
    # the cold lookups the sort took plus the lookups of the hot rows make
    # up the batch (hot rows are never sorted, cold ones always)
    if name != "hot_full":
        hot_keys = np.concatenate(hot) if hot else np.zeros(0, np.int64)
        is_hot = np.isin(sel.astype(np.int64), hot_keys)
        assert int(cnt[is_hot].sum()) + n_cold == w.n
        assert not np.isin(uk, hot_keys).any()
