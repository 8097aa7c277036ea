"""Seeded synthetic TBE inputs shaped like the workloads the pages describe.

This module only draws random numbers and lays them out; it holds none of the
TBE arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle (tests)
take their inputs from here, so that both sides see identical arrays.

Recipes (all seeded; per-table streams use seed * 1000 + t):
  tiny      T=2, E=1000, D=(64,128), B=64, L=8, uniform rows, int64
  small     T=1, E=64, D=128, B=65536, L=128, uniform rows, int64
  mixed     T=32, E=round(exp U(ln 1e4, ln 1e6)), D from {32,64,96,128,256},
            B=4096, L=min(Poisson(20), 200), Zipf(1.05) rows, int64
  weighted  T=64, E=round(exp U(ln 1e3, ln 5e6)), D from {16,32,64,128,160},
            B=8192, L uniform in {1..100}, Zipf(1.2) rows, psw U(0,1), int32
  hot       T=8, E=1e7, D=128, B=131072, L=200, Zipf(1.4) rows, int64
Weights are N(0, 0.01^2) rounded to fp16, momentum starts at 0, grad_out is
N(0, 1) fp32, lr = 0.01, eps = 1e-8.  Zipf(alpha) draws rank k in 1..E_t with
probability proportional to k^-alpha by inverse CDF of the truncated
distribution, then maps rank k to row perm_t[k-1] of a seeded random
permutation of the table's rows.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class Spec:
    name: str
    T: int
    B: int
    E: object            # int, or ("loguniform", lo, hi)
    D: object            # tuple of per-table widths, or ("choice", (...))
    L: object            # int (fixed), ("poisson", mean, max) or ("uniform", lo, hi)
    rows: object         # "uniform" or ("zipf", alpha)
    weighted: bool = False
    index_dtype: torch.dtype = torch.int64
    lr: float = 0.01
    eps: float = 1e-8


SPECS = {
    "tiny": Spec("tiny", T=2, B=64, E=1000, D=(64, 128), L=8, rows="uniform"),
    "small": Spec("small", T=1, B=65536, E=64, D=(128,), L=128, rows="uniform"),
    "mixed": Spec("mixed", T=32, B=4096, E=("loguniform", 1e4, 1e6),
                  D=("choice", (32, 64, 96, 128, 256)), L=("poisson", 20.0, 200),
                  rows=("zipf", 1.05)),
    "weighted": Spec("weighted", T=64, B=8192, E=("loguniform", 1e3, 5e6),
                     D=("choice", (16, 32, 64, 128, 160)), L=("uniform", 1, 100),
                     rows=("zipf", 1.2), weighted=True, index_dtype=torch.int32),
    "hot": Spec("hot", T=8, B=131072, E=10_000_000, D=(128,) * 8, L=200, rows=("zipf", 1.4)),
}


@dataclass
class Workload:
    name: str
    T: int
    B: int
    E: np.ndarray            # int64 [T] rows per table
    D: np.ndarray            # int64 [T] widths
    indices: torch.Tensor    # [n] int32/int64
    offsets: torch.Tensor    # [T*B+1], same dtype as indices, table-major bags
    psw: torch.Tensor | None # [n] fp32 or None
    weights: torch.Tensor    # flat fp16 or bf16, table t rows contiguous with stride D_t
    momentum: torch.Tensor   # fp32 [sum E]
    grad_out: torch.Tensor   # fp32 [B, sum D]
    lr: float
    eps: float
    extra: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return int(self.indices.numel())

    def to(self, device) -> "Workload":
        mv = lambda x: None if x is None else x.to(device)
        return Workload(self.name, self.T, self.B, self.E, self.D, mv(self.indices),
                        mv(self.offsets), mv(self.psw), mv(self.weights), mv(self.momentum),
                        mv(self.grad_out), self.lr, self.eps, dict(self.extra))


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _table_sizes(spec: Spec, T: int, seed: int):
    rng = np.random.default_rng(seed)
    if isinstance(spec.E, tuple):
        _, lo, hi = spec.E
        E = np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), size=T))).astype(np.int64)
    else:
        E = np.full(T, int(spec.E), dtype=np.int64)
    if spec.D[0] == "choice":
        D = rng.choice(np.asarray(spec.D[1], dtype=np.int64), size=T)
    else:
        D = np.asarray(spec.D[:T], dtype=np.int64)
    return E, D.astype(np.int64)


def _lengths(spec: Spec, B: int, g, device):
    if isinstance(spec.L, int):
        return torch.full((B,), spec.L, dtype=torch.int64, device=device)
    kind = spec.L[0]
    if kind == "poisson":
        lam = torch.full((B,), float(spec.L[1]), dtype=torch.float64, device=device)
        return torch.poisson(lam, generator=g).clamp_(0, spec.L[2]).to(torch.int64)
    if kind == "uniform":
        return torch.randint(spec.L[1], spec.L[2] + 1, (B,), generator=g, device=device)
    raise ValueError(kind)


def zipf_cdf(E: int, alpha: float, device):
    """Cumulative distribution of the truncated Zipf law P(k) ~ k^-alpha, k=1..E.
    Summed on the host in a fixed order (a parallel device scan may round
    differently from run to run), then moved to `device`."""
    k = torch.arange(1, E + 1, dtype=torch.float64)
    c = torch.cumsum(k.pow_(-alpha), 0)
    return c.div_(c[-1].clone()).to(device)


def _rows(spec: Spec, E: int, count: int, g, device, gperm=None):
    """Rows of `count` lookups.  Zipf ranks are drawn from g and mapped
    through a random permutation of the table's rows, drawn from gperm when
    given (a table seed of its own, so batches with other draw seeds share
    the table's row popularity) and else from g after the ranks."""
    if count == 0:
        return torch.zeros(0, dtype=torch.int64, device=device)
    if spec.rows == "uniform":
        return torch.randint(0, E, (count,), generator=g, device=device)
    _, alpha = spec.rows
    cdf = zipf_cdf(E, alpha, device)
    u = torch.rand(count, dtype=torch.float64, generator=g, device=device)
    rank = torch.searchsorted(cdf, u, right=True).clamp_(max=E - 1)
    perm = torch.randperm(E, generator=gperm if gperm is not None else g, device=device)
    return perm[rank]


def _lookups(spec: Spec, T: int, B: int, E, device, seed: int, table_seed: int | None):
    """Bag lengths, rows and per-sample weights of one batch, per table."""
    lengths, rows, psws = [], [], []
    for t in range(T):
        g = _gen(device, seed * 1000 + t)
        gperm = None if table_seed is None else _gen(device, table_seed * 1000 + 500 + t)
        L = _lengths(spec, B, g, device)
        cnt = int(L.sum().item())
        lengths.append(L)
        rows.append(_rows(spec, int(E[t]), cnt, g, device, gperm))
        if spec.weighted:
            psws.append(torch.rand(cnt, dtype=torch.float32, generator=g, device=device))
    return lengths, rows, psws


def _csr(spec: Spec, T: int, B: int, lengths, rows, device):
    L = torch.cat(lengths)
    offsets = torch.zeros(T * B + 1, dtype=torch.int64, device=device)
    torch.cumsum(L, 0, out=offsets[1:])
    return torch.cat(rows).to(spec.index_dtype), offsets.to(spec.index_dtype)


def make(name: str, device="cpu", seed: int = 0, B: int | None = None, T: int | None = None,
         E_scale: float | None = None, compact: bool = False,
         weights_dtype: torch.dtype = torch.float16, table_seed: int | None = None) -> Workload:
    """Draw a workload.  B, T and E_scale shrink a recipe for oracle-sized tests
    (E_scale multiplies every table's row count, keeping at least one row).
    compact=True keeps only the rows the lookups touch, renumbered per table
    in increasing order (the lookups are drawn from the full tables first), so
    that a few bags of a huge table need no huge weight array.  weights_dtype
    (torch.float16 or torch.bfloat16) is the type the N(0, 0.01^2) weight
    draws are stored in.  table_seed, when given, seeds the tables (sizes and
    each table's row permutation) apart from the batch draws, so that
    workloads of one table_seed and different seeds are distinct batches over
    the same tables (see batch()); without it both come from seed."""
    spec = SPECS[name]
    T = spec.T if T is None else T
    B = spec.B if B is None else B
    device = torch.device(device)
    E, D = _table_sizes(spec, T, seed if table_seed is None else table_seed)
    if E_scale is not None:
        E = np.maximum(1, np.rint(E * E_scale)).astype(np.int64)
    lengths, rows, psws = _lookups(spec, T, B, E, device, seed, table_seed)
    if compact:
        for t in range(T):
            uniq, inv = torch.unique(rows[t], return_inverse=True)
            rows[t] = inv
            E[t] = max(1, int(uniq.numel()))
    indices, offsets = _csr(spec, T, B, lengths, rows, device)
    psw = torch.cat(psws) if spec.weighted else None
    gw = _gen(device, seed * 1000 + 999)
    nW = int((E * D).sum())
    weights = torch.empty(nW, dtype=weights_dtype, device=device)
    chunk = 1 << 27
    for s in range(0, nW, chunk):
        e = min(nW, s + chunk)
        weights[s:e] = (torch.randn(e - s, generator=gw, device=device) * 0.01).to(weights_dtype)
    momentum = torch.zeros(int(E.sum()), dtype=torch.float32, device=device)
    grad_out = torch.randn(B, int(D.sum()), generator=gw, device=device)
    return Workload(name, T, B, E, D, indices, offsets, psw, weights, momentum, grad_out,
                    spec.lr, spec.eps, dict(table_seed=table_seed))


def batch(w: Workload, seed: int) -> Workload:
    """Another batch over the tables of w (drawn with a table_seed): new
    bags, lookups, per-sample weights and gradients from `seed`, the same
    tables, row popularity, weights and momentum (shared tensors, not
    copies)."""
    table_seed = w.extra.get("table_seed")
    if table_seed is None:
        raise ValueError("batch() needs a workload drawn with a table_seed")
    spec = SPECS[w.name]
    device = w.indices.device
    lengths, rows, psws = _lookups(spec, w.T, w.B, w.E, device, seed, table_seed)
    indices, offsets = _csr(spec, w.T, w.B, lengths, rows, device)
    psw = torch.cat(psws) if spec.weighted else None
    gw = _gen(device, seed * 1000 + 998)
    grad_out = torch.randn(w.B, int(w.D.sum()), generator=gw, device=device)
    return Workload(w.name, w.T, w.B, w.E, w.D, indices, offsets, psw, w.weights, w.momentum,
                    grad_out, w.lr, w.eps, dict(w.extra))


def from_arrays(E, D, B, indices, offsets, weights, grad_out, psw=None, momentum=None,
                lr=0.01, eps=1e-8, name="custom") -> Workload:
    """Wrap hand-made arrays (numpy or torch, on the host) as a Workload
    (weights: fp16; a bfloat16 tensor or float32 weights are kept as they
    are)."""
    t = lambda x, dt=None: None if x is None else torch.as_tensor(np.asarray(x) if not
                                                                   torch.is_tensor(x) else x,
                                                                   dtype=dt)
    E = np.asarray(E, dtype=np.int64)
    D = np.asarray(D, dtype=np.int64)
    idx = t(indices)
    off = t(offsets, idx.dtype)
    m = t(momentum, torch.float32) if momentum is not None else torch.zeros(int(E.sum()))
    if torch.is_tensor(weights) and weights.dtype in (torch.bfloat16, torch.float32):
        W = weights
    elif not torch.is_tensor(weights) and np.asarray(weights).dtype == np.float32:
        W = t(weights, torch.float32)
    else:
        W = t(weights, torch.float16)
    return Workload(name, len(E), int(B), E, D, idx, off, t(psw, torch.float32), W, m,
                    t(grad_out, torch.float32), lr, eps)
