"""The seeded input generator (host only): each recipe has the shapes, value
ranges and structure the workload list states (tables, widths, bag-length
laws, row laws, index type, per-sample weights), draws are reproducible, and
batches drawn over one table seed share their tables and row popularity."""
import math

import numpy as np
import pytest
import torch

import workloads

# reduced sizes (B, T, E_scale) that keep every recipe's structure
REDUCED = {
    "tiny": dict(),
    "small": dict(B=4096),
    "mixed": dict(B=2048, E_scale=0.1),
    "weighted": dict(B=1024, T=16, E_scale=0.01),
    "hot": dict(B=512, T=2, E_scale=0.01),
}


def _np(x):
    return None if x is None else x.numpy()


@pytest.mark.parametrize("name", list(REDUCED))
def test_recipe_shapes_and_ranges(name):
    spec = workloads.SPECS[name]
    kw = REDUCED[name]
    w = workloads.make(name, seed=3, **kw)
    T, B = w.T, w.B
    assert T == kw.get("T", spec.T) and B == kw.get("B", spec.B)
    assert w.indices.dtype == spec.index_dtype and w.offsets.dtype == spec.index_dtype
    off = _np(w.offsets).astype(np.int64)
    assert off.shape == (T * B + 1,) and off[0] == 0 and off[-1] == w.n
    L = np.diff(off)
    assert np.all(L >= 0)
    idx = _np(w.indices).astype(np.int64)
    for t in range(T):
        rows = idx[off[t * B]:off[(t + 1) * B]]
        assert rows.size == 0 or (rows.min() >= 0 and rows.max() < w.E[t])
    # widths and table sizes
    if spec.D[0] == "choice":
        assert set(w.D.tolist()) <= set(spec.D[1])
    else:
        assert w.D.tolist() == list(spec.D[:T])
    scale = kw.get("E_scale", 1.0)
    if isinstance(spec.E, tuple):
        _, lo, hi = spec.E
        assert np.all(w.E >= math.floor(lo * scale)) and np.all(w.E <= math.ceil(hi * scale))
    else:
        assert np.all(w.E == max(1, round(spec.E * scale)))
    # bag lengths
    if isinstance(spec.L, int):
        assert np.all(L == spec.L)
    elif spec.L[0] == "poisson":
        assert L.max() <= spec.L[2] and abs(L.mean() - spec.L[1]) < 0.1
    else:
        assert L.min() >= spec.L[1] and L.max() <= spec.L[2]
        assert abs(L.mean() - (spec.L[1] + spec.L[2]) / 2) < 1.0
    # per-sample weights, state and gradients
    if spec.weighted:
        p = _np(w.psw)
        assert p.shape == (w.n,) and p.dtype == np.float32 and p.min() >= 0 and p.max() < 1
    else:
        assert w.psw is None
    assert w.weights.dtype == torch.float16 and w.weights.numel() == int((w.E * w.D).sum())
    assert abs(float(w.weights.float().std()) - 0.01) < 0.001
    assert w.momentum.shape == (int(w.E.sum()),) and not w.momentum.any()
    assert w.grad_out.shape == (B, int(w.D.sum())) and w.grad_out.dtype == torch.float32
    assert (w.lr, w.eps) == (spec.lr, spec.eps)


@pytest.mark.parametrize("name", ["mixed", "weighted"])
def test_draws_are_reproducible(name):
    a = workloads.make(name, seed=5, **REDUCED[name])
    b = workloads.make(name, seed=5, **REDUCED[name])
    c = workloads.make(name, seed=6, **REDUCED[name])
    for x, y in ((a.indices, b.indices), (a.offsets, b.offsets), (a.weights, b.weights),
                 (a.grad_out, b.grad_out)):
        assert torch.equal(x, y)
    assert np.array_equal(a.E, b.E) and np.array_equal(a.D, b.D)
    if a.psw is not None:
        assert torch.equal(a.psw, b.psw)
    assert not (a.indices.numel() == c.indices.numel() and torch.equal(a.indices, c.indices))


def test_batches_over_one_table_seed_share_tables_and_popularity():
    kw = REDUCED["hot"]
    w0 = workloads.make("hot", seed=1, table_seed=7, **kw)
    w1 = workloads.batch(w0, seed=2)
    w2 = workloads.make("hot", seed=2, table_seed=7, **kw)
    # batch() draws what make() draws for that seed over the same tables
    assert torch.equal(w1.indices, w2.indices) and torch.equal(w1.offsets, w2.offsets)
    assert np.array_equal(w1.E, w0.E) and w1.weights is w0.weights
    assert not torch.equal(w1.indices, w0.indices)
    # Zipf(1.4): the most looked-up row of each table is the same row
    B = w0.B
    for t in range(w0.T):
        top = []
        for w in (w0, w1):
            off = w.offsets.numpy()
            rows = w.indices.numpy()[off[t * B]:off[(t + 1) * B]]
            top.append(np.bincount(rows, minlength=int(w.E[t])).argmax())
        assert top[0] == top[1]
    with pytest.raises(ValueError):
        workloads.batch(workloads.make("tiny", seed=0), seed=1)


def test_zipf_draws_follow_the_truncated_law():
    # ranks drawn by inverse CDF: the k-th most frequent row's share matches
    # k^-alpha / H(E, alpha) within five standard deviations
    E, alpha, n = 20, 1.4, 400_000
    spec = workloads.Spec("z", T=1, B=1, E=E, D=(8,), L=1, rows=("zipf", alpha))
    g = torch.Generator().manual_seed(11)
    rows = workloads._rows(spec, E, n, g, torch.device("cpu")).numpy()
    freq = np.sort(np.bincount(rows, minlength=E))[::-1] / n
    k = np.arange(1, E + 1, dtype=np.float64)
    p = k ** -alpha / (k ** -alpha).sum()
    sd = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(freq - p) < 5 * sd + 1e-12)
    cdf = workloads.zipf_cdf(E, alpha, "cpu").numpy()
    assert cdf[-1] == 1.0 and np.all(np.diff(cdf) > 0)


def test_compact_renumbers_touched_rows_in_order():
    kw = dict(B=64, E_scale=0.01)
    full = workloads.make("mixed", seed=4, **kw)
    comp = workloads.make("mixed", seed=4, compact=True, **kw)
    assert torch.equal(full.offsets, comp.offsets)
    off = full.offsets.numpy()
    B = full.B
    for t in range(full.T):
        a = full.indices.numpy()[off[t * B]:off[(t + 1) * B]]
        b = comp.indices.numpy()[off[t * B]:off[(t + 1) * B]]
        uniq, inv = np.unique(a, return_inverse=True)
        assert np.array_equal(b, inv) and comp.E[t] == max(1, uniq.size)
