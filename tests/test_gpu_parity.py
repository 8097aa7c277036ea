"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Sizes are chosen so the oracle finishes in seconds while the GPU kernels
still run many sort tiles, many bags per table, ragged last tiles, short and
long runs and multi-level reduction trees."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

# (recipe, overrides) -- reduced so the oracle runs in seconds
CASES = {
    "tiny": dict(name="tiny"),
    "small": dict(name="small", B=4096),
    "mixed": dict(name="mixed", B=512, E_scale=0.05),
    "weighted": dict(name="weighted", B=256, E_scale=0.02),
    "hot": dict(name="hot", B=1024, E_scale=0.01),
}


def make(case, seed=0):
    kw = dict(CASES[case])
    return workloads.make(kw.pop("name"), seed=seed, **kw)


def oracle_forward(w, hw):
    tab = H.tables(w)
    ref = oracle.forward(tab, w.B, hw["weights"], hw["indices"], hw["offsets"], hw["psw"])
    absw = np.abs(hw["weights"])
    absp = None if hw["psw"] is None else np.abs(hw["psw"])
    terms = oracle.forward(tab, w.B, absw, hw["indices"], hw["offsets"], absp)
    return ref, terms


@pytest.mark.parametrize("case", list(CASES))
def test_forward_matches_oracle(case):
    w = make(case)
    hw = H.host(w)
    run = H.Run(w)
    out = run.forward(flags=0)
    ref, terms = oracle_forward(w, hw)
    H.assert_forward_close(out, ref, terms)
    out2 = run.forward(flags=H.tbe.TBE_F_FORCE_GENERIC)
    H.assert_forward_close(out2, ref, terms)


@pytest.mark.parametrize("case", list(CASES))
def test_preprocess_bit_exact(case):
    w = make(case)
    hw = H.host(w)
    run = H.Run(w)
    got = run.preprocess()
    ref = oracle.preprocess(H.tables(w), w.B, hw["indices"], hw["offsets"])
    nv = len(ref["sorted_keys"])
    assert got["n_valid"] == nv
    assert got["R"] == len(ref["unique_keys"])
    assert np.array_equal(got["sorted_keys"][:nv], ref["sorted_keys"])
    assert np.array_equal(got["sorted_bags"][:nv], ref["sorted_bags"])
    assert np.array_equal(got["unique_keys"], ref["unique_keys"])
    assert np.array_equal(got["run_starts"].astype(np.int64), ref["run_starts"])
    if hw["psw"] is not None:
        assert np.array_equal(got["sorted_psw"][:nv], hw["psw"][ref["sorted_pos"]])
    # pairs: a new pair wherever the key or the bag changes
    ps, pb, rp = H.pair_structure(ref["sorted_keys"], ref["sorted_bags"], ref["run_starts"])
    assert got["P"] == len(pb)
    assert np.array_equal(got["pair_starts"].astype(np.int64), ps)
    assert np.array_equal(got["pair_bags"].astype(np.int64), pb)
    assert np.array_equal(got["run_pairs"].astype(np.int64), rp)
    # device-side classification: exactly the runs of at least long_threshold pairs
    npairs = np.diff(rp)
    exp_long = np.nonzero(npairs >= got["long_threshold"])[0]
    assert np.array_equal(np.sort(got["long_runs"]), exp_long)
    chunk = got["chunk"]
    assert got["n_chunks"] == int(((npairs[exp_long] + chunk - 1) // chunk).sum())


@pytest.mark.parametrize("two_launch", [False, True])
@pytest.mark.parametrize("case", list(CASES))
def test_backward_matches_oracle(case, two_launch):
    w = make(case)
    rng = np.random.default_rng(5)
    # a nonzero starting accumulator exercises m_old + mean(g^2)
    w.momentum = torch.from_numpy(rng.uniform(0, 0.5, int(w.E.sum())).astype(np.float32))
    hw = H.host(w)
    run = H.Run(w)
    flags = H.tbe.TBE_F_LONG_TWO_LAUNCH if two_launch else 0
    W_gpu, m_gpu = run.backward(flags)
    tab = H.tables(w)
    W_ref, m_ref = oracle.backward_rowwise_adagrad(tab, w.B, hw["indices"], hw["offsets"],
                                                   hw["grad_out"], hw["weights"], hw["momentum"],
                                                   w.lr, w.eps, hw["psw"])
    H.assert_momentum_close(m_gpu, m_ref)
    H.assert_weights_within_ulp(W_gpu, W_ref)
    # untouched rows: bit-identical weights and momentum
    keys, _ = oracle.row_gradients(tab, w.B, hw["indices"], hw["offsets"], hw["grad_out"],
                                   hw["psw"])
    touched = np.zeros(int(w.E.sum()), bool)
    touched[keys] = True
    assert np.array_equal(m_gpu[~touched].view(np.uint32), hw["momentum"][~touched].view(np.uint32))
    wmask = H.row_mask(tab, keys)
    assert np.array_equal(W_gpu[~wmask].view(np.uint16), hw["weights"][~wmask].view(np.uint16))
    assert run.status() == 0


def test_two_steps_accumulate():
    w = make("mixed", seed=3)
    hw = H.host(w)
    run = H.Run(w)
    tab = H.tables(w)
    W_ref, m_ref = hw["weights"], hw["momentum"]
    steps = []
    for _ in range(2):
        run.backward()
        W_ref, m_ref = oracle.backward_rowwise_adagrad(tab, w.B, hw["indices"], hw["offsets"],
                                                       hw["grad_out"], W_ref, m_ref, w.lr, w.eps)
        steps.append(W_ref)
    W_gpu, m_gpu = run.weights.cpu().numpy(), run.momentum.cpu().numpy()
    H.assert_momentum_close(m_gpu, m_ref)
    # A 1-ulp difference allowed after the first step is carried into the
    # second, where the weight may have moved to a smaller binade: bound the
    # gap by one ulp of each step's oracle value.
    ulp = lambda x: np.spacing(np.abs(x).astype(np.float16)).astype(np.float64)
    tol = ulp(steps[0]) + ulp(steps[1])
    err = np.abs(W_gpu.astype(np.float64) - W_ref.astype(np.float64))
    assert not (err > tol).any(), f"{(err > tol).sum()} weights beyond the two-step bound"


def test_int32_and_int64_indices_agree():
    w = make("mixed", seed=4)
    run64 = H.Run(w)
    out64 = run64.forward()
    W64, m64 = run64.backward()
    w32 = workloads.from_arrays(w.E, w.D, w.B, w.indices.to(torch.int32), w.offsets.to(torch.int32),
                                w.weights, w.grad_out, lr=w.lr, eps=w.eps)
    run32 = H.Run(w32)
    assert np.array_equal(run32.forward(), out64)
    W32, m32 = run32.backward()
    assert np.array_equal(W32.view(np.uint16), W64.view(np.uint16))
    assert np.array_equal(m32.view(np.uint32), m64.view(np.uint32))


def test_launch_counter_counts_the_kernels_of_a_call():
    # tiny: two tables, so the generic forward is one kernel; with bounds
    # checking the offsets check adds one more
    w = make("tiny")
    run = H.Run(w)
    c0 = H.tbe.tbe_kernel_launches()
    run.forward(flags=0)
    c1 = H.tbe.tbe_kernel_launches()
    run.forward(flags=H.tbe.TBE_F_CHECK_BOUNDS)
    c2 = H.tbe.tbe_kernel_launches()
    run.preprocess()
    c3 = H.tbe.tbe_kernel_launches()
    assert c1 - c0 == 1
    assert c2 - c1 == 2
    assert c3 - c2 >= 10  # expand, sort passes, run-length encoding, classify


def test_probe_times_the_selected_kernel():
    w = make("hot")
    run = H.Run(w)
    run.backward()  # warm-up: module load, hot set
    H.tbe.tbe_probe_set(H.tbe.TBE_PROBE_LONG_CHUNKS)
    run.backward()
    run.backward()
    launches, ms = H.tbe.tbe_probe_read()
    H.tbe.tbe_probe_set(H.tbe.TBE_PROBE_OFF)
    assert launches == 2 and ms > 0.0
    run.backward()
    assert H.tbe.tbe_probe_read() == (0, 0.0)  # switched off
