"""Pins for the CPU oracle: the worked example printed on the HugeCTR page,
closed forms, special cases that reduce to library routines, brute force on
tiny inputs, and invariants.  None of these re-type the oracle's code."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.conftest import load_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --------------------------------------------------------------- fp16 codec
def test_half_to_double_matches_numpy_for_every_bit_pattern(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_double_to_half_matches_numpy_rounding(oracle_lib):
    rng = np.random.default_rng(1)
    halves = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (halves[:-1] + halves[1:]) / 2          # exact ties: nearest-even decides
    vals = np.concatenate([
        halves, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1),
        rng.normal(0, 0.01, 20000), rng.normal(0, 100, 5000),
        np.ldexp(rng.uniform(0.5, 1, 5000), rng.integers(-30, 17, 5000)),
        [65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26, 0.0, -0.0],
    ])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------- HugeCTR worked example
def test_preprocess_matches_hugectr_worked_example(oracle_lib):
    g = load_golden("hugectr_worked_example.txt")
    tab = oracle.Tables([g["E"][0]], [8])
    idx = np.array(g["rows"], np.int64)
    off = np.array(g["offsets"], np.int64)
    pp = oracle.preprocess(tab, g["B"][0], idx, off)
    assert pp["sorted_keys"].tolist() == g["sorted_rows"]
    assert pp["sorted_bags"].tolist() == g["sorted_bags"]
    assert pp["run_starts"].tolist() == g["run_starts"]
    assert len(pp["unique_keys"]) == g["count"][0]
    # The page's intermediate arrays agree with the oracle's runs: a flag marks
    # each run start, and its inclusive prefix sum numbers the runs.
    flags = [int(i in pp["run_starts"][:-1]) for i in range(len(idx))]
    assert flags == g["flags"]
    assert np.cumsum(flags).tolist() == g["flag_scan"]
    # The sample id of every sorted lookup, read through the sort permutation,
    # is its bag: the expansion step of the page.
    assert [g["sample_id"][p] for p in pp["sorted_pos"]] == g["sorted_bags"]
    # keys -> rows by the tens digit, as the page maps them
    assert [k // 10 for k in g["keys"]] == g["rows"]


# ------------------------------------------------------------- random cases
def _tiny_problem(seed, T=3, B=5, maxL=6, E=(7, 4, 9), D=(8, 16, 8), weighted=False,
                  dtype=np.int64, invalid=False):
    rng = np.random.default_rng(seed)
    E = np.asarray(E[:T]); D = np.asarray(D[:T])
    L = rng.integers(0, maxL + 1, T * B)
    off = np.concatenate([[0], np.cumsum(L)]).astype(dtype)
    idx = np.concatenate([rng.integers(0, E[t], L[t * B:(t + 1) * B].sum()) for t in range(T)])
    if invalid and len(idx):
        bad = rng.random(len(idx)) < 0.15
        idx[bad] = rng.choice([-1, -7, 10 ** 6], bad.sum())
    idx = idx.astype(dtype)
    tab = oracle.Tables(E, D)
    W = (rng.normal(0, 0.5, int((E * D).sum()))).astype(np.float16)
    G = rng.normal(0, 1, (B, int(D.sum()))).astype(np.float32)
    psw = rng.uniform(0, 1, len(idx)).astype(np.float32) if weighted else None
    return tab, B, idx, off, W, G, psw


def _lookups(tab, B, idx, off):
    """(t, b, position, row) for every lookup, read straight from the CSR arrays."""
    out = []
    for bag in range(tab.T * B):
        t, b = divmod(bag, B)
        for i in range(int(off[bag]), int(off[bag + 1])):
            out.append((t, b, i, int(idx[i])))
    return out


@pytest.mark.parametrize("seed", range(6))
def test_preprocess_brute_force(oracle_lib, seed):
    tab, B, idx, off, *_ = _tiny_problem(seed, invalid=seed % 2 == 1)
    pp = oracle.preprocess(tab, B, idx, off)
    look = [(int(tab.hash_base[t]) + r, b, i) for t, b, i, r in _lookups(tab, B, idx, off)
            if 0 <= r < tab.E[t]]
    keys = sorted({k for k, _, _ in look})
    # O(n * R): for each key in increasing order, list its lookups by position.
    exp_keys, exp_bags, exp_pos, starts = [], [], [], []
    for k in keys:
        starts.append(len(exp_keys))
        for kk, b, i in sorted(look, key=lambda x: x[2]):
            if kk == k:
                exp_keys.append(k); exp_bags.append(b); exp_pos.append(i)
    starts.append(len(exp_keys))
    assert pp["sorted_keys"].tolist() == exp_keys
    assert pp["sorted_bags"].tolist() == exp_bags
    assert pp["sorted_pos"].tolist() == exp_pos
    assert pp["unique_keys"].tolist() == keys
    assert pp["run_starts"].tolist() == starts
    # invariants: sum of run lengths = number of valid lookups; keys strictly increase
    assert int(np.diff(pp["run_starts"]).sum()) == len(look)
    assert np.all(np.diff(pp["unique_keys"].astype(np.int64)) > 0)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("weighted", [False, True])
def test_forward_brute_force_exact_rational(oracle_lib, seed, weighted):
    tab, B, idx, off, W, G, psw = _tiny_problem(seed, weighted=weighted, dtype=np.int32,
                                                invalid=seed == 3)
    out = oracle.forward(tab, B, W, idx, off, psw)
    exp = np.zeros_like(out, dtype=object)
    exp[:] = Fraction(0)
    for t, b, i, r in _lookups(tab, B, idx, off):
        if not 0 <= r < tab.E[t]:
            continue
        c = Fraction(float(psw[i])) if weighted else Fraction(1)
        base = int(tab.w_offsets[t]) + r * int(tab.D[t])
        for d in range(int(tab.D[t])):
            exp[b, int(tab.D_offsets[t]) + d] += c * Fraction(float(W[base + d]))
    exact = np.array([[float(x) for x in row] for row in exp])
    # the double sum is rounded once to fp32: within half an fp32 ulp of exact
    ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(out.astype(np.float64) - exact) <= 0.5 * ulp + 1e-300)


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("weighted", [False, True])
def test_pool_gathered_exact_and_equal_to_forward(oracle_lib, seed, weighted):
    """pool_gathered (the checker of the full-size forward tests) pools rows
    that the caller gathered itself.  Against the definition: each bag's sum,
    computed in exact rationals from rows gathered here with numpy and
    rounded once to fp32.  And bit for bit against oracle.forward on the same
    bags.  Bags are ragged (lengths 0..9, never equal to D, some empty) and
    every coefficient differs, so an offset coefficient or a row stride of
    the wrong length changes the result."""
    tab, B, idx, off, W, G, psw = _tiny_problem(seed, weighted=weighted, dtype=np.int64)
    rng = np.random.default_rng(100 + seed)
    # re-draw ragged bags over table 0 only
    T, D = 1, int(tab.D[0])
    tab1 = oracle.Tables([int(tab.E[0])], [D])
    lens = rng.integers(0, 10, B)
    lens[1] = 0
    off1 = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    n = int(off1[-1])
    idx1 = rng.integers(0, int(tab.E[0]), n).astype(np.int64)
    W1 = W[:int(tab.E[0]) * D]
    coef = rng.uniform(0.1, 2.0, n).astype(np.float32) if weighted else None
    rows = W1.reshape(-1, D)[idx1]                      # gathered here, by numpy
    got = oracle.pool_gathered(off1, rows, coef)
    assert got.shape == (B, D)
    for b in range(B):
        for d in range(D):
            acc = Fraction(0)
            for i in range(off1[b], off1[b + 1]):
                c = Fraction(float(coef[i])) if weighted else Fraction(1)
                acc += c * Fraction(float(rows[i, d]))
            exact = float(acc)
            ulp = float(np.spacing(np.float32(abs(exact))))
            assert abs(float(got[b, d]) - exact) <= 0.5 * ulp + 1e-300, (b, d)
    ref = oracle.forward(tab1, B, W1, idx1, off1, coef)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_forward_closed_forms(oracle_lib):
    tab = oracle.Tables([5, 3], [8, 16])
    rng = np.random.default_rng(0)
    W = rng.normal(0, 1, int(tab.w_offsets[-1])).astype(np.float16)
    B = 4
    # table 0: bag0 one-hot row 2; bag1 row 4 repeated 2048 times; bag2 empty; bag3 rows 0,1
    # table 1: bag0 one-hot row 1; bag1 empty; bag2 row 2 x3; bag3 row 0
    bags = [[2], [4] * 2048, [], [0, 1], [1], [], [2, 2, 2], [0]]
    idx = np.array([r for bg in bags for r in bg], np.int64)
    off = np.concatenate([[0], np.cumsum([len(b) for b in bags])]).astype(np.int64)
    out = oracle.forward(tab, B, W, idx, off)
    row = lambda t, r: W[tab.w_offsets[t] + r * tab.D[t]: tab.w_offsets[t] + (r + 1) * tab.D[t]]
    assert np.array_equal(out[0, :8], row(0, 2).astype(np.float32))
    assert np.array_equal(out[1, :8], 2048 * row(0, 4).astype(np.float32))
    assert np.array_equal(out[2, :8], np.zeros(8, np.float32))
    assert np.array_equal(out[0, 8:], row(1, 1).astype(np.float32))
    assert np.array_equal(out[1, 8:], np.zeros(16, np.float32))
    assert np.array_equal(out[2, 8:], 3 * row(1, 2).astype(np.float32))
    # a per-sample weight scales its single row: one rounding of an exact product
    psw = np.full(len(idx), 1.0, np.float32)
    assert np.array_equal(oracle.forward(tab, B, W, idx, off, psw), out)
    psw[0] = 0.3
    o2 = oracle.forward(tab, B, W, idx, off, psw)
    assert np.array_equal(o2[0, :8],
                          (np.float64(np.float32(0.3)) * row(0, 2).astype(np.float64))
                          .astype(np.float32))


def test_forward_skips_out_of_range_rows(oracle_lib):
    tab, B, idx, off, W, G, psw = _tiny_problem(11)
    bad_idx = idx.copy()
    bad_idx[::5] = -3
    keep = np.ones(len(idx), bool)
    keep[::5] = False
    # drop those lookups from the CSR by hand
    new_off = np.array([keep[:o].sum() for o in off], np.int64)
    assert np.array_equal(oracle.forward(tab, B, W, bad_idx, off),
                          oracle.forward(tab, B, W, idx[keep], new_off))


# ------------------------------------------------------------------ backward
def _single_row_problem(D, grad_row, w0, m0=0.0, lr=0.01, eps=1e-8, reps=1, E=3, row=1):
    tab = oracle.Tables([E], [D])
    W = np.zeros(E * D, np.float16)
    W[row * D:(row + 1) * D] = w0
    m = np.zeros(E, np.float32)
    m[row] = m0
    G = np.asarray(grad_row, np.float32).reshape(1, D)
    idx = np.array([row] * reps, np.int64)
    off = np.array([0, reps], np.int64)
    W2, m2 = oracle.backward_rowwise_adagrad(tab, 1, idx, off, G, W, m, lr, eps)
    return W2.reshape(E, D), m2


@pytest.mark.parametrize("c", [0.75, -2.5, 1e-3])
@pytest.mark.parametrize("eps", [1e-8, 0.5])
def test_adagrad_constant_gradient_closed_form(oracle_lib, c, eps):
    # g_d = c for all d, m0 = 0:  m = mean(c^2) = c^2,  w -= lr*c/(|c| + eps)
    D, lr = 12, 0.01
    w0 = np.float16(0.125)
    W2, m2 = _single_row_problem(D, [c] * D, w0, lr=lr, eps=eps)
    c32 = np.float64(np.float32(c))          # the gradient is stored in fp32
    assert m2[1] == np.float32(c32 * c32)
    exp = np.float16(float(w0) - np.float64(np.float32(lr)) * c32 /
                     (np.sqrt(np.float64(np.float32(c32 * c32))) + np.float64(np.float32(eps))))
    assert np.all(W2[1] == exp)
    assert np.all(W2[0] == 0) and np.all(W2[2] == 0) and m2[0] == 0 and m2[2] == 0
    # eps under the square root would give a different value when eps is large
    if eps == 0.5 and abs(c) >= 0.5:
        inside = np.float16(float(w0) - lr * c / np.sqrt(c * c + eps))
        assert inside != exp


def test_adagrad_second_step_accumulates(oracle_lib):
    # from m0 = c^2 with the same gradient: m = 2c^2, step = lr*c/(sqrt(2)|c| + eps)
    D, c, lr, eps = 8, 1.5, 0.05, 1e-8
    W2, m2 = _single_row_problem(D, [c] * D, np.float16(1.0), m0=c * c, lr=lr, eps=eps)
    assert m2[1] == np.float32(2 * c * c)
    exp = np.float16(1.0 - lr * c / (np.sqrt(np.float64(np.float32(2 * c * c))) + eps))
    assert np.all(W2[1] == exp)


def test_adagrad_mean_uses_true_width(oracle_lib):
    # half the entries c, half 0 over D=6: mean(g^2) = c^2/2; zero entries keep w
    c = 2.0
    W2, m2 = _single_row_problem(6, [c, c, c, 0, 0, 0], np.float16(0.5), lr=0.1)
    assert m2[1] == np.float32(c * c / 2)
    exp = np.float16(0.5 - 0.1 * c / (c / np.sqrt(2.0) + np.float64(np.float32(1e-8))))
    assert np.all(W2[1, :3] == exp) and np.all(W2[1, 3:] == np.float16(0.5))


def test_adagrad_D1_equals_elementwise_hugectr_rule(oracle_lib):
    # For D = 1 the row mean is the element itself, so row-wise Adagrad equals the
    # element-wise rule of the HugeCTR Adagrad kernel: acc += g*g; w -= lr*g/(sqrt(acc)+eps).
    rng = np.random.default_rng(3)
    lr, eps = 0.05, 1e-3
    tab = oracle.Tables([4], [1])
    W = rng.normal(0, 1, 4).astype(np.float16)
    m = np.zeros(4, np.float32)
    acc = np.zeros(4, np.float64)
    w_el = W.astype(np.float64)
    for step in range(4):
        idx = rng.integers(0, 4, 6).astype(np.int64)
        off = np.array([0, 2, 6], np.int64)
        G = rng.normal(0, 1, (2, 1)).astype(np.float32)
        W, m = oracle.backward_rowwise_adagrad(tab, 2, idx, off, G, W, m, lr, eps)
        g = np.zeros(4)
        for i, r in enumerate(idx):
            g[r] += G[0 if i < 2 else 1, 0]
        for r in range(4):
            if (idx == r).any():
                acc[r] = np.float32(acc[r] + g[r] * g[r])
                w_el[r] = np.float16(w_el[r] - lr * g[r] / (np.sqrt(acc[r]) + np.float32(eps)))
        assert np.array_equal(m.astype(np.float64), acc)
        assert np.array_equal(W, w_el.astype(np.float16))


def test_duplicate_rows_in_a_bag_count_per_occurrence(oracle_lib):
    # The page's example: a slot "30,20,20,20" updates row 2 with three copies of
    # the bag gradient and row 3 with one.
    tab = oracle.Tables([6], [4])
    G = np.array([[1.0, -2.0, 0.5, 3.0]], np.float32)
    idx = np.array([3, 2, 2, 2], np.int64)
    off = np.array([0, 4], np.int64)
    keys, g = oracle.row_gradients(tab, 1, idx, off, G)
    assert keys.tolist() == [2, 3]
    assert np.array_equal(g[0], 3 * G[0].astype(np.float64))
    assert np.array_equal(g[1], G[0].astype(np.float64))


@pytest.mark.parametrize("seed", range(4))
def test_row_gradients_brute_force_exact(oracle_lib, seed):
    tab, B, idx, off, W, G, psw = _tiny_problem(seed + 20, weighted=True, invalid=seed == 1)
    keys, g = oracle.row_gradients(tab, B, idx, off, G, psw)
    exp = {}
    for t, b, i, r in _lookups(tab, B, idx, off):
        if not 0 <= r < tab.E[t]:
            continue
        k = int(tab.hash_base[t]) + r
        D = int(tab.D[t])
        row = exp.setdefault(k, [Fraction(0)] * D)
        for d in range(D):
            row[d] += Fraction(float(psw[i])) * Fraction(float(G[b, int(tab.D_offsets[t]) + d]))
    assert keys.tolist() == sorted(exp)
    for j, k in enumerate(keys):
        e = np.array([float(x) for x in exp[int(k)]])
        assert np.allclose(g[j, :len(e)], e, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_backward_invariants(oracle_lib, seed):
    tab, B, idx, off, W, G, psw = _tiny_problem(seed + 40, weighted=seed % 2 == 0)
    rng = np.random.default_rng(seed)
    m0 = rng.uniform(0, 2, int(tab.hash_base[-1])).astype(np.float32)
    W2, m2 = oracle.backward_rowwise_adagrad(tab, B, idx, off, G, W, m0, 0.01, 1e-8, psw)
    keys, g = oracle.row_gradients(tab, B, idx, off, G, psw)
    touched = np.zeros(int(tab.hash_base[-1]), bool)
    touched[keys] = True
    # untouched rows: weights and momentum bit-identical
    for t in range(tab.T):
        D, E = int(tab.D[t]), int(tab.E[t])
        for r in range(E):
            k = int(tab.hash_base[t]) + r
            sl = slice(int(tab.w_offsets[t]) + r * D, int(tab.w_offsets[t]) + (r + 1) * D)
            if not touched[k]:
                assert W2[sl].view(np.uint16).tolist() == W[sl].view(np.uint16).tolist()
                assert m2[k].view(np.uint32) == m0[k].view(np.uint32)
    # every touched row updated exactly once: the momentum increment is the mean
    # square of the row's summed gradient (per-lookup updates would differ)
    for j, k in enumerate(keys):
        t = int(np.searchsorted(tab.hash_base, k, side="right") - 1)
        D = int(tab.D[t])
        inc = np.mean(g[j, :D] ** 2)
        assert abs(float(m2[k]) - (float(m0[k]) + inc)) <= 2e-7 * (float(m0[k]) + inc)
    # gradient mass: summed over runs equals summed over lookups
    mass_runs = sum(g[j, :int(tab.D[np.searchsorted(tab.hash_base, k, side='right') - 1])].sum()
                    for j, k in enumerate(keys))
    mass_lookups = 0.0
    for t, b, i, r in _lookups(tab, B, idx, off):
        c = psw[i] if psw is not None else 1.0
        mass_lookups += float(c) * float(
            G[b, int(tab.D_offsets[t]):int(tab.D_offsets[t + 1])].astype(np.float64).sum())
    assert abs(mass_runs - mass_lookups) <= 1e-9 * max(1.0, abs(mass_lookups))


def test_backward_selected_agrees_with_full(oracle_lib):
    tab, B, idx, off, W, G, psw = _tiny_problem(77, weighted=True)
    m0 = np.linspace(0, 1, int(tab.hash_base[-1])).astype(np.float32)
    W2, m2 = oracle.backward_rowwise_adagrad(tab, B, idx, off, G, W, m0, 0.02, 1e-6, psw)
    maxD = int(tab.D.max())
    sel = np.arange(int(tab.hash_base[-1]), dtype=np.uint32)
    w_rows = np.zeros((len(sel), maxD), np.float16)
    for k in sel:
        t = int(np.searchsorted(tab.hash_base, k, side="right") - 1)
        D = int(tab.D[t]); r = int(k) - int(tab.hash_base[t])
        w_rows[k, :D] = W[tab.w_offsets[t] + r * D: tab.w_offsets[t] + (r + 1) * D]
    ws, ms, cnt = oracle.backward_selected(tab, B, idx, off, G, 0.02, 1e-6, sel, w_rows, m0[sel],
                                           psw)
    assert np.array_equal(ms.view(np.uint32), m2[sel].view(np.uint32))
    for k in sel:
        t = int(np.searchsorted(tab.hash_base, k, side="right") - 1)
        D = int(tab.D[t]); r = int(k) - int(tab.hash_base[t])
        assert np.array_equal(ws[k, :D].view(np.uint16),
                              W2[tab.w_offsets[t] + r * D: tab.w_offsets[t] + (r + 1) * D]
                              .view(np.uint16))
    assert int(cnt.sum()) == len(idx)


def test_repair_offsets_examples(oracle_lib):
    # first entry forced to 0, entries clamped to [0, n], then made non-decreasing
    got, changed = oracle.repair_offsets(np.array([3, 5, 3, 12, 8], np.int64), 10)
    assert got.tolist() == [0, 5, 5, 10, 10] and changed == 4
    got, changed = oracle.repair_offsets(np.array([0, -4, 2, 2, 9], np.int32), 9)
    assert got.tolist() == [0, 0, 2, 2, 9] and changed == 1
    ok = np.array([0, 1, 1, 4], np.int64)
    got, changed = oracle.repair_offsets(ok, 4)
    assert got.tolist() == ok.tolist() and changed == 0


def test_oracle_rejects_bad_offsets(oracle_lib):
    tab = oracle.Tables([4], [8])
    with pytest.raises(ValueError):
        oracle.forward(tab, 2, np.zeros(32, np.float16), np.zeros(3, np.int64),
                       np.array([0, 2, 1], np.int64))


# -------------------------------------------------------------- mean pooling
# HugeCTR page, combiner note and mean backward kernel: with mean pooling a
# bag of L > 1 lookups is scaled by 1/L (L by the row offsets), bags of 0 or 1
# lookups are not scaled, and the backward scales the bag's gradient before
# the regrouping.
def test_mean_forward_of_identical_rows_is_the_row(oracle_lib):
    tab = oracle.Tables([6], [8])
    rng = np.random.default_rng(21)
    W = rng.normal(0, 1, 48).astype(np.float16)
    bags = [[3] * 7, [5], [], [0, 0, 0, 0]]
    idx = np.array([r for b in bags for r in b], np.int64)
    off = np.concatenate([[0], np.cumsum([len(b) for b in bags])]).astype(np.int64)
    out = oracle.forward(tab, 4, W, idx, off, mean=True)
    row = lambda r: W[r * 8:(r + 1) * 8].astype(np.float32)
    # 7 copies summed in double then divided by 7: the row exactly
    assert np.array_equal(out[0], row(3))
    assert np.array_equal(out[1], row(5))        # L = 1: unscaled
    assert np.array_equal(out[2], np.zeros(8, np.float32))
    assert np.array_equal(out[3], row(0))
    # and the sum pooling of the same bags is L times larger
    s = oracle.forward(tab, 4, W, idx, off)
    assert np.array_equal(s[0], (7 * W[24:32].astype(np.float64)).astype(np.float32))


def test_mean_counts_out_of_range_lookups_in_L(oracle_lib):
    # a bag [r, invalid] has L = 2: its mean is half the row; the invalid
    # lookup adds nothing but still counts
    tab = oracle.Tables([4], [8])
    W = np.arange(32, dtype=np.float16) / 8
    idx = np.array([1, 9], np.int64)
    off = np.array([0, 2], np.int64)
    out = oracle.forward(tab, 1, W, idx, off, mean=True)
    assert np.array_equal(out[0], (W[8:16].astype(np.float64) / 2).astype(np.float32))


@pytest.mark.parametrize("L", [1, 2, 5, 64])
def test_mean_backward_of_one_bag_equals_the_single_lookup_update(oracle_lib, L):
    # one bag of L lookups of one row: the row's gradient is L * g / L = g,
    # the update of a single (sum-pooled) lookup of that row
    D = 16
    rng = np.random.default_rng(L)
    g = rng.normal(0, 1, D).astype(np.float32)
    w0 = rng.normal(0, 0.1, D).astype(np.float16)
    tab = oracle.Tables([3], [D])
    W = np.zeros(3 * D, np.float16)
    W[D:2 * D] = w0
    m = np.full(3, 0.25, np.float32)
    G = g.reshape(1, D)
    W1, m1 = oracle.backward_rowwise_adagrad(tab, 1, np.array([1] * L, np.int64),
                                             np.array([0, L], np.int64), G, W, m, 0.05, 1e-8,
                                             mean=True)
    W2, m2 = oracle.backward_rowwise_adagrad(tab, 1, np.array([1], np.int64),
                                             np.array([0, 1], np.int64), G, W, m, 0.05, 1e-8)
    if L in (1, 2, 64):  # L * (g / L) is exact for powers of two
        assert np.array_equal(W1, W2) and np.array_equal(m1, m2)
    else:
        assert np.allclose(m1, m2, rtol=1e-6)
        assert np.max(np.abs(W1.astype(np.float64) - W2.astype(np.float64))) <= \
            np.max(np.spacing(np.abs(W2.astype(np.float16)))).astype(np.float64)


@pytest.mark.parametrize("seed", range(3))
def test_mean_gradients_equal_sum_gradients_of_scaled_grad_out(oracle_lib, seed):
    # scaling each bag's grad_out row by its L and pooling with mean gives the
    # sum-pooling gradients (L a power of two: every product exact)
    rng = np.random.default_rng(40 + seed)
    E, D, B = [9, 5], [8, 16], 6
    T = 2
    lens = rng.choice([0, 1, 2, 4, 8], size=T * B)
    idx = np.concatenate([rng.integers(0, E[t], int(lens[t * B + b]))
                          for t in range(T) for b in range(B)]).astype(np.int64)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tab = oracle.Tables(E, D)
    G = rng.normal(0, 1, (B, sum(D))).astype(np.float32)
    Gs = G.copy()
    for t in range(T):
        d0 = int(tab.D_offsets[t])
        for b in range(B):
            L = int(lens[t * B + b])
            if L > 1:
                Gs[b, d0:d0 + D[t]] *= L
    k1, g1 = oracle.row_gradients(tab, B, idx, off, Gs, mean=True)
    k2, g2 = oracle.row_gradients(tab, B, idx, off, G)
    assert np.array_equal(k1, k2)
    assert np.array_equal(g1, g2)


# ------------------------------------------------------------- bf16 weights
def test_bf16_to_double_matches_torch_for_every_bit_pattern(oracle_lib):
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.int64).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_double_to_bf16_matches_torch_rounding(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    fin = np.arange(0, 0x7f80, dtype=np.int64).astype(np.uint16)
    vals16 = torch.from_numpy(fin.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    mids = ((vals16[:-1].astype(np.float64) + vals16[1:]) / 2).astype(np.float32)  # exact ties
    vals = np.concatenate([
        vals16, mids, -mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1)),
        rng.normal(0, 0.01, 20000).astype(np.float32), rng.normal(0, 1e30, 2000).astype(np.float32),
        np.float32([3.3895314e38, 3.3961775e38, 3.4e38, 1e-40, 1e-45, 0.0, -0.0]),
    ]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.double_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("seed", range(3))
def test_forward_bf16_brute_force_exact_rational(oracle_lib, seed):
    tab, B, idx, off, W, G, psw = _tiny_problem(seed, weighted=True, dtype=np.int64)
    rng = np.random.default_rng(100 + seed)
    Wb = rng.integers(0, 0x7f00, len(W)).astype(np.uint16) | \
        (rng.integers(0, 2, len(W)).astype(np.uint16) << 15)
    Wb &= np.uint16(0xbfff)  # keep exponents moderate (top exponent bit clear)
    out = oracle.forward(tab, B, Wb, idx, off, psw, bf16=True)
    exp = np.zeros_like(out, dtype=object)
    exp[:] = Fraction(0)
    for t, b, i, r in _lookups(tab, B, idx, off):
        if not 0 <= r < tab.E[t]:
            continue
        c = Fraction(float(psw[i]))
        base = int(tab.w_offsets[t]) + r * int(tab.D[t])
        for d in range(int(tab.D[t])):
            exp[b, int(tab.D_offsets[t]) + d] += c * Fraction(oracle.bf16_to_double(int(Wb[base + d])))
    exact = np.array([[float(x) for x in row] for row in exp])
    ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(out.astype(np.float64) - exact) <= 0.5 * ulp + 1e-300)


@pytest.mark.parametrize("c", [0.75, -2.5])
def test_adagrad_bf16_constant_gradient_closed_form(oracle_lib, c):
    torch = pytest.importorskip("torch")
    D, lr, eps = 12, 0.01, 1e-8
    tab = oracle.Tables([3], [D])
    w0 = oracle.double_to_bf16(0.125)
    W = np.zeros(3 * D, np.uint16)
    W[D:2 * D] = w0
    m = np.zeros(3, np.float32)
    G = np.full((1, D), c, np.float32)
    W2, m2 = oracle.backward_rowwise_adagrad(tab, 1, np.array([1], np.int64), np.array([0, 1]),
                                             G, W, m, lr, eps, bf16=True)
    c32 = np.float64(np.float32(c))
    assert m2[1] == np.float32(c32 * c32)
    step = 0.125 - lr * c32 / (np.sqrt(np.float64(np.float32(c32 * c32))) + eps)
    # closed form rounded by the oracle; where the double step is an fp32
    # value, torch's fp32 -> bf16 rounding must give the same bits
    ref = torch.tensor([step], dtype=torch.float64).float().to(torch.bfloat16)
    want = oracle.double_to_bf16(step)
    assert np.all(W2[D:2 * D] == want)
    assert np.all(W2[:D] == 0) and np.all(W2[2 * D:] == 0)
    # the rounding agrees with torch's where the fp32 value is exact
    if np.float64(np.float32(step)) == step:
        assert int(ref.view(torch.int16).item()) & 0xffff == want


# ------------------------------------------------ element-wise Adagrad
# HugeCTR's Adagrad kernel keeps one accumulator per weight element:
# acc_d += g_d^2, w_d -= lr * g_d / (sqrt(acc_d) + eps).  The oracle's
# element-wise mode keeps that accumulator at the weight's own flat position.

def _elementwise_row_problem(D, v, K, w0, m0, lr, eps, E=3, row=1):
    """K identical bags, each looking up `row` once with gradient row v."""
    tab = oracle.Tables([E], [D])
    W = np.zeros(E * D, np.float16)
    W[row * D:(row + 1) * D] = w0
    m = np.zeros(E * D, np.float32)
    m[row * D:(row + 1) * D] = m0
    G = np.tile(np.asarray(v, np.float32), (K, 1))
    idx = np.full(K, row, np.int64)
    off = np.arange(K + 1, dtype=np.int64)
    W2, m2 = oracle.backward_rowwise_adagrad(tab, K, idx, off, G, W, m, lr, eps,
                                             elementwise=True)
    return W2.reshape(E, D), m2.reshape(E, D)


def test_elementwise_first_step_with_eps_zero_moves_each_element_by_lr():
    # From acc = 0 with eps = 0 the step is lr * g/|g| = lr * sign(g) for every
    # element, whatever its magnitude; acc becomes g^2 with g = K v (exact).
    v = np.array([3.0, -0.015625, 1e-3, -250.0, 0.5, -7.25, 40.0, -1.0], np.float32)
    K, lr = 3, 0.125
    W2, m2 = _elementwise_row_problem(8, v, K, np.float16(0.5), 0.0, lr, 0.0)
    assert np.array_equal(W2[1], np.where(v > 0, np.float16(0.375), np.float16(0.625)))
    g = K * v.astype(np.float64)
    assert np.array_equal(m2[1], (g * g).astype(np.float32))
    # other rows untouched, their accumulators too
    assert not W2[0].any() and not W2[2].any() and not m2[0].any() and not m2[2].any()


def test_elementwise_second_step_divides_by_sqrt_two():
    # From acc = g^2 with the same gradient: acc = 2 g^2, step = lr/sqrt(2)
    v = np.array([2.0, -0.25, 64.0, -3.0, 0.75, -1e-2, 9.0, -5.5], np.float32)
    lr = 0.125
    g2 = (v.astype(np.float64)) ** 2
    W2, m2 = _elementwise_row_problem(8, v, 1, np.float16(0.375), g2.astype(np.float32), lr, 0.0)
    assert np.array_equal(m2[1], (2 * g2).astype(np.float32))
    exp = (0.375 - np.sign(v) * lr / np.sqrt(2.0)).astype(np.float16)
    assert np.array_equal(W2[1], exp)


def test_elementwise_equals_rowwise_when_every_element_has_the_same_magnitude():
    # |g_d| = c for all d: the row mean of g^2 is c^2, the element-wise
    # accumulators all equal it, and the two rules give the same step.
    D, c, lr, eps = 16, 0.375, 0.05, 1e-3
    v = np.where(np.arange(D) % 3 == 0, -c, c).astype(np.float32)
    W_el, m_el = _elementwise_row_problem(D, v, 2, np.float16(0.25), 0.5, lr, eps)
    W_rw, m_rw = _single_row_problem(D, 2 * v, np.float16(0.25), m0=0.5, lr=lr, eps=eps)
    assert np.array_equal(W_el, W_rw)
    assert np.array_equal(m_el[1], np.full(D, m_rw[1], np.float32))


def test_elementwise_D1_equals_rowwise():
    # For D = 1 the two rules coincide (the row-wise D = 1 case is pinned to
    # the HugeCTR rule above), over several steps and per-sample weights.
    rng = np.random.default_rng(11)
    tab = oracle.Tables([5, 3], [1, 1])
    W = rng.normal(0, 1, 8).astype(np.float16)
    m = rng.uniform(0, 1, 8).astype(np.float32)
    We, me, Wr, mr = W.copy(), m.copy(), W.copy(), m.copy()
    for step in range(3):
        idx = np.concatenate([rng.integers(0, 5, 7), rng.integers(0, 3, 5)]).astype(np.int64)
        off = np.array([0, 3, 7, 9, 12], np.int64)
        G = rng.normal(0, 1, (2, 2)).astype(np.float32)
        psw = rng.uniform(0.5, 2, 12).astype(np.float32)
        We, me = oracle.backward_rowwise_adagrad(tab, 2, idx, off, G, We, me, 0.05, 1e-3, psw,
                                                 elementwise=True)
        Wr, mr = oracle.backward_rowwise_adagrad(tab, 2, idx, off, G, Wr, mr, 0.05, 1e-3, psw)
        assert np.array_equal(We, Wr) and np.array_equal(me, mr)


@pytest.mark.parametrize("seed", range(3))
def test_elementwise_invariants(oracle_lib, seed):
    # untouched elements bit-identical; each touched element's accumulator
    # grows by exactly its own summed gradient squared, once
    tab, B, idx, off, W, G, psw = _tiny_problem(seed + 70, weighted=seed != 1)
    rng = np.random.default_rng(seed)
    nW = int(tab.w_offsets[-1])
    m0 = rng.uniform(0, 2, nW).astype(np.float32)
    W2, m2 = oracle.backward_rowwise_adagrad(tab, B, idx, off, G, W, m0, 0.01, 1e-8, psw,
                                             elementwise=True)
    keys, g = oracle.row_gradients(tab, B, idx, off, G, psw)
    touched = np.zeros(nW, bool)
    for j, k in enumerate(keys):
        t = int(np.searchsorted(tab.hash_base, k, side="right") - 1)
        D = int(tab.D[t])
        s = int(tab.w_offsets[t]) + (int(k) - int(tab.hash_base[t])) * D
        touched[s:s + D] = True
        exp = m0[s:s + D].astype(np.float64) + g[j, :D] ** 2
        assert np.all(np.abs(m2[s:s + D] - exp) <= 2 ** -23 * exp)
    assert np.array_equal(W2.view(np.uint16)[~touched], W.view(np.uint16)[~touched])
    assert np.array_equal(m2.view(np.uint32)[~touched], m0.view(np.uint32)[~touched])
    assert (W2.view(np.uint16)[touched] != W.view(np.uint16)[touched]).any()


def test_elementwise_momentum_must_be_shaped_like_the_weights():
    tab = oracle.Tables([4], [8])
    with pytest.raises(ValueError):
        oracle.backward_rowwise_adagrad(tab, 1, np.array([1]), np.array([0, 1]),
                                        np.ones((1, 8), np.float32), np.zeros(32, np.float16),
                                        np.zeros(4, np.float32), 0.1, 1e-8, elementwise=True)


# -------------------------------------------------------------- fp32 weights
# The FBTriton page pools fp32 weights in fp64.  The oracle reads fp32
# weights exactly, sums in double and rounds the result once.

@pytest.mark.parametrize("seed", range(3))
def test_forward_fp32_brute_force_exact_rational(oracle_lib, seed):
    # fp32 weights with full 24-bit significands (not representable in 16-bit
    # types); the exact rational sum rounded once to fp32 is the answer
    tab, B, idx, off, W, G, psw = _tiny_problem(seed + 60, weighted=seed != 2)
    rng = np.random.default_rng(200 + seed)
    Wf = (rng.standard_normal(len(W)) * (1 + rng.random(len(W)) * 2.0 ** -12)).astype(np.float32)
    out = oracle.forward(tab, B, Wf, idx, off, psw, fp32=True)
    exp = np.zeros_like(out, dtype=object)
    exp[:] = Fraction(0)
    for t, b, i, r in _lookups(tab, B, idx, off):
        if not 0 <= r < tab.E[t]:
            continue
        c = Fraction(float(psw[i])) if psw is not None else Fraction(1)
        base = int(tab.w_offsets[t]) + r * int(tab.D[t])
        for d in range(int(tab.D[t])):
            exp[b, int(tab.D_offsets[t]) + d] += c * Fraction(float(Wf[base + d]))
    exact = np.array([[float(x) for x in row] for row in exp])
    ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(out.astype(np.float64) - exact) <= 0.5 * ulp + 1e-300)
    # the 16-bit readings of the same bits would not give this result
    assert not np.array_equal(out, oracle.forward(tab, B, Wf.astype(np.float16), idx, off, psw))


@pytest.mark.parametrize("elementwise", [False, True])
def test_adagrad_fp32_keeps_full_precision(oracle_lib, elementwise):
    # From m = 0 with eps = 0 and a row of equal |g|, both Adagrad forms step
    # every element by exactly lr against the sign of g.  w0 = 1 + 2^-20 and
    # lr = 2^-10 make w0 -+ lr exact in fp32 but not in fp16 or bf16.
    D = 8
    tab = oracle.Tables([3], [D])
    w0 = np.float32(1 + 2.0 ** -20)
    W = np.full(3 * D, np.float32(0.3), np.float32)
    W[D:2 * D] = w0
    m = np.zeros(3 * D if elementwise else 3, np.float32)
    v = np.array([0.5, -0.5, 0.5, 0.5, -0.5, -0.5, 0.5, -0.5], np.float32)
    W2, m2 = oracle.backward_rowwise_adagrad(tab, 1, np.array([1], np.int64), np.array([0, 1]),
                                             v.reshape(1, D), W, m, 2.0 ** -10, 0.0,
                                             elementwise=elementwise, fp32=True)
    assert W2.dtype == np.float32
    exp = np.where(v > 0, 1 + 2.0 ** -20 - 2.0 ** -10, 1 + 2.0 ** -20 + 2.0 ** -10)
    assert np.array_equal(W2[D:2 * D].astype(np.float64), exp)
    # untouched rows keep their (non-16-bit) values bit for bit
    assert np.array_equal(W2[:D].view(np.uint32), W[:D].view(np.uint32))
    assert np.array_equal(W2[2 * D:].view(np.uint32), W[2 * D:].view(np.uint32))


def test_backward_fp32_agrees_with_fp16_on_fp16_values_when_nothing_rounds():
    # Weights and steps that are exact in fp16 give the same result whichever
    # type holds them: w0 = 0.5, lr = 0.125, eps = 0, |g| equal in the row.
    D = 16
    tab = oracle.Tables([2], [D])
    rng = np.random.default_rng(4)
    v = np.where(rng.random(D) < 0.5, -2.0, 2.0).astype(np.float32).reshape(1, D)
    W16 = np.full(2 * D, np.float16(0.5))
    W16[:D] = np.float16(0.25)
    args = (tab, 1, np.array([1], np.int64), np.array([0, 1]), v)
    Wa, ma = oracle.backward_rowwise_adagrad(*args, W16, np.zeros(2, np.float32), 0.125, 0.0)
    Wb, mb = oracle.backward_rowwise_adagrad(*args, W16.astype(np.float32),
                                             np.zeros(2, np.float32), 0.125, 0.0, fp32=True)
    assert np.array_equal(Wa.astype(np.float32), Wb) and np.array_equal(ma, mb)


def test_elementwise_closed_form_with_bf16_weights_and_mean_pooling():
    # One bag looking up row 1 three times, mean pooling: the row's gradient is
    # 3 x (1/3) x grad_out = grad_out (exactly 1 in double only up to
    # rounding of 1/3; eps = 0 makes the step lr * sign(g) regardless).  bf16
    # weights 0.5 and lr = 0.125 keep 0.375 / 0.625 exact.
    D = 8
    tab = oracle.Tables([3], [D])
    w0 = oracle.double_to_bf16(0.5)
    W = np.full(3 * D, w0, np.uint16)
    m = np.zeros(3 * D, np.float32)
    v = np.array([[1.5, -0.25, 4.0, -8.0, 0.5, -1.0, 2.0, -3.0]], np.float32)
    W2, m2 = oracle.backward_rowwise_adagrad(tab, 1, np.array([1, 1, 1], np.int64),
                                             np.array([0, 3]), v, W, m, 0.125, 0.0, mean=True,
                                             bf16=True, elementwise=True)
    want = [oracle.double_to_bf16(0.375 if x > 0 else 0.625) for x in v[0]]
    assert W2[D:2 * D].tolist() == want
    assert np.allclose(m2[D:2 * D], v[0].astype(np.float64) ** 2, rtol=2 ** -22)
    assert (W2[:D] == w0).all() and (W2[2 * D:] == w0).all() and not m2[:D].any()
