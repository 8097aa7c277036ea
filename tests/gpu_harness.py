"""Helpers for tests that run the CUDA path and the oracle on the same inputs.

Inputs come from workloads (seeded); the CUDA path is reached only through
the C-ABI binding; the oracle only through oracle/.  Nothing here computes a
TBE result itself.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import table_embedding_bag_gb300 as tbe


def ws_array(ws, ptr, count, dtype=torch.int32):
    """Copy `count` 4-byte elements at device address ptr (inside ws) to numpy."""
    off = ptr - ws.buf.data_ptr()
    assert 0 <= off and off + 4 * count <= ws.nbytes
    a = ws.buf[off:off + 4 * count].view(dtype).cpu().numpy()
    return a.view(np.uint32) if dtype == torch.int32 else a


def host(w):
    """Host numpy copies of a workload's arrays (psw None when unweighted)."""
    t = lambda x: None if x is None else x.detach().cpu().numpy()
    return dict(indices=t(w.indices), offsets=t(w.offsets), psw=t(w.psw), weights=t(w.weights),
                momentum=t(w.momentum), grad_out=t(w.grad_out))


class Run:
    """One TBE problem on the GPU through the C ABI."""

    def __init__(self, w, device="cuda", mean=False, weights_dtype=torch.float16,
                 elementwise=False):
        self.w = w
        self.ew_flag = tbe.TBE_F_ELEMENTWISE if elementwise else 0
        self.desc = tbe.TBEDesc(w.E, w.D, w.B, w.indices.dtype, device, weights_dtype)
        self.ws = tbe.Workspace(self.desc, max(w.n, 1), w.psw is not None, device, mean=mean)
        d = lambda x: None if x is None else x.to(device).contiguous()
        self.indices, self.offsets, self.psw = d(w.indices), d(w.offsets), d(w.psw)
        self.weights = d(w.weights).clone()
        assert self.weights.dtype == weights_dtype, "the workload's weights have another dtype"
        self.momentum = d(w.momentum).clone()
        self.grad_out = d(w.grad_out)
        self.out = torch.empty(w.B, self.desc.total_D, dtype=torch.float32, device=device)

    def forward(self, flags=0):
        tbe.tbe_forward(self.desc, self.weights, self.indices, self.offsets, self.psw, self.out,
                        self.ws, flags)
        torch.cuda.synchronize()
        return self.out.cpu().numpy()

    def preprocess(self, flags=0):
        tbe.tbe_preprocess(self.desc, self.indices, self.offsets, self.psw, self.ws, flags)
        torch.cuda.synchronize()
        v = tbe.tbe_workspace_view(self.desc, max(self.w.n, 1), self.ws)
        counts = ws_array(self.ws, v["counts"], 8)
        R, nv, P = int(counts[0]), int(counts[1]), int(counts[6])
        res = dict(R=R, n_valid=nv, n_long=int(counts[2]), n_chunks=int(counts[3]), P=P,
                   run_pairs=ws_array(self.ws, v["run_pairs"], R + 1),
                   pair_starts=ws_array(self.ws, v["pair_starts"], P + 1),
                   pair_bags=ws_array(self.ws, v["pair_bags"], P),
                   sorted_keys=ws_array(self.ws, v["sorted_keys"], self.w.n),
                   sorted_bags=ws_array(self.ws, v["sorted_bags"], self.w.n),
                   unique_keys=ws_array(self.ws, v["unique_keys"], R),
                   run_starts=ws_array(self.ws, v["run_starts"], R + 1),
                   long_runs=ws_array(self.ws, v["long_runs"], int(counts[2])),
                   long_threshold=v["long_threshold"], chunk=v["chunk"])
        if v["sorted_psw"]:
            res["sorted_psw"] = ws_array(self.ws, v["sorted_psw"], self.w.n, torch.float32)
        return res

    def backward(self, flags=0):
        tbe.tbe_backward_rowwise_adagrad(self.desc, self.grad_out, self.indices, self.offsets,
                                         self.psw, self.weights, self.momentum, self.w.lr,
                                         self.w.eps, self.ws, flags | self.ew_flag)
        torch.cuda.synchronize()
        return self.host_weights(), self.momentum.cpu().numpy()

    def host_weights(self):
        """The weights on the host: fp16 values, or bf16 bit patterns (uint16)."""
        if self.weights.dtype == torch.bfloat16:
            return bf16_bits(self.weights)
        return self.weights.cpu().numpy()

    def status(self):
        return tbe.tbe_read_status(self.ws)

    def hot_set(self):
        """The workspace's hot rows: list (per table) of sorted linear keys."""
        torch.cuda.synchronize()
        v = tbe.tbe_workspace_view(self.desc, max(self.w.n, 1), self.ws)
        T, K = self.desc.T, v["hot_slots"]
        n = ws_array(self.ws, v["hot_n"], T)
        keys = ws_array(self.ws, v["hot_keys"], T * K).reshape(T, K)
        return [keys[t, :n[t]].astype(np.int64) for t in range(T)]

    def reset_state(self):
        """Weights and momentum back to the workload's values."""
        self.weights.copy_(self.w.weights.to(self.weights.device))
        self.momentum.copy_(self.w.momentum.to(self.momentum.device))


def tables(w):
    return oracle.Tables(w.E, w.D)


# ------------------------------------------------------------- comparisons
def assert_forward_close(out, ref, abs_terms, rel=1e-5):
    """|out - ref| <= rel * sum|terms| elementwise (sum|terms| from the oracle on |W|, |psw|)."""
    err = np.abs(out.astype(np.float64) - ref.astype(np.float64))
    tol = rel * abs_terms.astype(np.float64) + 1e-30
    bad = err > tol
    assert not bad.any(), (f"{bad.sum()} of {bad.size} forward outputs off; worst err "
                           f"{err.max():.3e} at {np.unravel_index(np.argmax(err - tol), err.shape)}")


def assert_momentum_close(m, ref, rel=1e-5):
    err = np.abs(m.astype(np.float64) - ref.astype(np.float64))
    tol = rel * np.abs(ref.astype(np.float64)) + 1e-30
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} momentum values off; worst rel {np.max(err / (tol / rel)):.3e}"


def bf16_bits(t):
    """A bfloat16 tensor's bit patterns as numpy uint16."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits):
    """bf16 bit patterns as float64 (a bf16 is the upper half of an fp32)."""
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_bf16_step_close(bits, ref_bits, old_bits, upd_rel=2.0 ** -12, max_frac=1e-5):
    """bf16 weights after an Adagrad step against the oracle's.  The kernel
    forms w - lr*g/(sqrt(m)+eps) in fp32 and rounds once to bf16; the oracle
    does the same in fp64.  Where the step nearly cancels the weight the
    result is far smaller than its operands, and because bf16 keeps fp32's
    exponent range (fp16 bottoms out at 2^-24) its ulp there can be below the
    fp32 error of the operands.  So each weight must lie within 1 ulp of the
    oracle's or within the fp32 error budget of the operands: 2^-12 of the
    step (an fp32 gradient summed over runs of up to a few thousand pairs,
    then divided) plus 2^-23 of the old weight; and at most max_frac of all
    weights may need more than the 1 ulp."""
    a, b = bf16_values(bits), bf16_values(ref_bits)
    old = bf16_values(old_bits)
    assert np.isfinite(a).all()
    err = np.abs(a - b)
    ulp = np.spacing(np.abs(b).astype(np.float32)).astype(np.float64) * 65536.0
    beyond = err > ulp
    tol = ulp + upd_rel * np.abs(old - b) + 2.0 ** -23 * np.abs(old)
    bad = err > tol
    worst = int(np.argmax(err - tol)) if err.size else 0
    detail = (f"{beyond.sum()} of {err.size} beyond 1 ulp, {bad.sum()} beyond the fp32 budget; "
              f"worst at {worst}: gpu {a[worst]:.9e} oracle {b[worst]:.9e} old {old[worst]:.9e}")
    print("bf16 step:", detail)
    assert not bad.any(), detail
    assert beyond.sum() <= max_frac * err.size, detail


def _touched_elements(tab, B, indices, offsets):
    """Per touched row (ascending linear key): its lookups' count, and the
    flat weight positions of its elements with their column numbers."""
    offsets = np.asarray(offsets, np.int64)
    idx = np.asarray(indices, np.int64)
    bag = np.repeat(np.arange(len(offsets) - 1), np.diff(offsets))
    t = bag // B
    E = np.asarray(tab.E, np.int64)
    ok = (idx >= 0) & (idx < E[t])
    keys = np.asarray(tab.hash_base, np.int64)[t[ok]] + idx[ok]
    ukeys, count = np.unique(keys, return_counts=True)
    kt = np.searchsorted(np.asarray(tab.hash_base, np.int64), ukeys, side="right") - 1
    D = np.asarray(tab.D, np.int64)[kt]
    base = np.asarray(tab.w_offsets, np.int64)[kt] + (ukeys - np.asarray(tab.hash_base)[kt]) * D
    row = np.repeat(np.arange(len(ukeys)), D)
    col = np.arange(row.size) - np.repeat(np.cumsum(D) - D, D)
    return ukeys, count, row, np.repeat(base, D) + col, col


def assert_elementwise_step_close(tab, B, indices, offsets, grad_out, psw, mean, lr, eps,
                                  w_old, m_old, w_gpu, m_gpu, w_ref, m_ref, bf16=False,
                                  max_loose=1e-3):
    """Element-wise Adagrad results against the oracle's, with an error bound
    derived from the arithmetic.  Each element's gradient g is an fp32 sum of
    n terms; whatever the order, it lies within d = (2 n + 10) 2^-24 S of the
    exact sum, S the sum of the terms' magnitudes (from the oracle on |grad|,
    |psw|): n - 1 additions (each within 2^-23 of its result, which also
    covers a tensor core's accumulator if it truncates rather than rounds),
    the products with per-sample weights and mean factors, and for hot rows
    the tensor-core products, whose split operands drop a remainder term of
    about 2^-21 of each product.  The accumulator m = m_old + g^2 is then off by at most
    (2|g| + d) d plus two fp32 roundings, and the step lr g / (sqrt(m) + eps)
    by what those two errors move it, plus its own fp32 rounding; the stored
    weight may differ by that plus one unit in the last place.  Touched
    elements must meet the bound, at most max_loose of them may need more
    than 1e-5 (momentum) or 1 ulp (weights), and untouched elements must be
    bit-identical to the inputs."""
    u = 2.0 ** -24
    ukeys, count, row, flat, col = _touched_elements(tab, B, indices, offsets)
    keys, g = oracle.row_gradients(tab, B, indices, offsets, grad_out, psw, mean)
    absp = None if psw is None else np.abs(psw)
    keys_a, S = oracle.row_gradients(tab, B, indices, offsets, np.abs(grad_out), absp, mean)
    assert np.array_equal(keys.astype(np.int64), ukeys) and np.array_equal(keys_a, keys)
    g = g[row, col]
    S = S[row, col]
    d = (2 * count[row] + 10) * u * S
    # momentum
    mr = m_ref[flat].astype(np.float64)
    mg = m_gpu[flat].astype(np.float64)
    dm = 4 * u * mr + (2 * np.abs(g) + d) * d
    bad = np.abs(mg - mr) > dm
    assert not bad.any(), f"{bad.sum()} of {flat.size} accumulators beyond the fp32 bound"
    loose = np.abs(mg - mr) > 1e-5 * mr
    assert loose.sum() <= max_loose * flat.size, f"{loose.sum()} accumulators beyond 1e-5"
    # weights
    if bf16:
        val = lambda x: bf16_values(x)
        spacing = lambda v: np.spacing(np.abs(v).astype(np.float32)).astype(np.float64) * 65536.0
    else:
        val = lambda x: np.asarray(x, np.float16).astype(np.float64)
        spacing = lambda v: np.spacing(np.abs(v).astype(np.float16)).astype(np.float64)
    wo = val(w_old)[flat]
    wr = val(w_ref)[flat]
    wg = val(w_gpu)[flat]
    lo = np.sqrt(np.maximum(mr - dm, 0.0)) + eps
    hi = np.sqrt(mr + dm) + eps
    step = lr * np.abs(g) / lo
    ds = lr * d / lo + lr * np.abs(g) * (1.0 / lo - 1.0 / hi) + 8 * u * step
    tol = ds + 2 * u * (np.abs(wo) + step) + np.maximum(spacing(wr), spacing(wg))
    err = np.abs(wg - wr)
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} of {flat.size} weights beyond the fp32 bound"
    loose = err > spacing(wr)
    assert loose.sum() <= max_loose * flat.size, f"{loose.sum()} weights beyond 1 ulp"
    # untouched elements unchanged
    mask = np.ones(np.asarray(m_gpu).size, bool)
    mask[flat] = False
    assert np.array_equal(np.asarray(m_gpu).view(np.uint32)[mask],
                          np.asarray(m_old, np.float32).view(np.uint32)[mask])
    assert np.array_equal(np.asarray(w_gpu).view(np.uint16)[mask],
                          np.asarray(w_old).view(np.uint16)[mask])
    print(f"element-wise step: {flat.size} touched elements; beyond 1e-5 / 1 ulp: "
          f"{int((np.abs(mg - mr) > 1e-5 * mr).sum())} / {int(loose.sum())}")


def assert_bf16_within_ulp(bits, ref_bits, ulps=1):
    """bf16 patterns within `ulps` steps of the oracle's (steps counted along
    the ordered sequence of finite bf16 values; +0 and -0 are the same step)."""
    def order(x):
        x = np.asarray(x, np.int64)
        return np.where(x & 0x8000, -(x & 0x7fff), x)
    a, b = np.asarray(bits, np.uint16), np.asarray(ref_bits, np.uint16)
    assert not np.isnan(bf16_values(a)).any() and not np.isinf(bf16_values(a)).any()
    bad = np.abs(order(a) - order(b)) > ulps
    assert not bad.any(), f"{bad.sum()} of {bad.size} bf16 weights beyond {ulps} ulp"


def assert_weights_within_ulp(w, ref, ulps=1):
    """fp16 values within `ulps` units in the last place of the oracle's value."""
    a = w.astype(np.float64)
    b = ref.astype(np.float64)
    ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    bad = np.abs(a - b) > ulps * ulp
    assert not bad.any(), f"{bad.sum()} of {bad.size} weights beyond {ulps} ulp"


def row_mask(tab, keys):
    """Boolean mask over the flat weights of the rows with the given linear keys."""
    mask = np.zeros(int(tab.w_offsets[-1]), bool)
    for k in np.asarray(keys, dtype=np.int64):
        t = int(np.searchsorted(tab.hash_base, k, side="right") - 1)
        r = int(k - tab.hash_base[t])
        D = int(tab.D[t])
        s = int(tab.w_offsets[t]) + r * D
        mask[s:s + D] = True
    return mask


def pair_structure(sorted_keys, sorted_bags, run_starts):
    """Pairs read off sorted arrays: a pair starts where the key or the bag
    changes.  Returns (pair_starts[P+1], pair_bags[P], run_pairs[R+1])."""
    k = np.asarray(sorted_keys, dtype=np.int64)
    b = np.asarray(sorted_bags, dtype=np.int64)
    n = len(k)
    head = np.ones(n, bool)
    if n:
        head[1:] = (k[1:] != k[:-1]) | (b[1:] != b[:-1])
    ps = np.concatenate([np.nonzero(head)[0], [n]]).astype(np.int64)
    rp = np.searchsorted(ps, np.asarray(run_starts, dtype=np.int64))
    return ps, b[ps[:-1]], rp


# ------------------------------------------------- sampled checks (any size)
def host_inputs(w):
    """indices, offsets, psw of a (device) workload as host numpy arrays."""
    return (w.indices.cpu().numpy(), w.offsets.cpu().numpy(),
            None if w.psw is None else w.psw.cpu().numpy())


def check_sampled_bags(w, weights_dev, out, nsample=300, seed=1, inputs=None):
    """Pooled outputs of sampled bags (the first, the last and `nsample`
    random ones) against oracle.pool_gathered on rows gathered from the
    device weights by index (no TBE arithmetic here)."""
    idx, off, psw = inputs if inputs is not None else host_inputs(w)
    rng = np.random.default_rng(seed)
    nb = w.T * w.B
    bags = np.unique(np.concatenate([[0, nb - 1], rng.integers(0, nb, nsample)]))
    D_off = np.concatenate([[0], np.cumsum(w.D)])
    W_off = np.concatenate([[0], np.cumsum(w.E * w.D)])
    checked = 0
    for t in np.unique(bags // w.B):
        tb = bags[bags // w.B == t]
        D = int(w.D[t])
        seg = [np.arange(off[b], off[b + 1]) for b in tb]
        pos = np.concatenate(seg) if seg else np.zeros(0, np.int64)
        rows = idx[pos].astype(np.int64)
        flat = torch.as_tensor(W_off[t] + rows[:, None] * D + np.arange(D)[None, :],
                               device=weights_dev.device)
        gathered = weights_dev[flat.reshape(-1)].reshape(len(rows), D).cpu().numpy()
        bo = np.concatenate([[0], np.cumsum([len(s) for s in seg])])
        coef = None if psw is None else psw[pos]
        ref = oracle.pool_gathered(bo, gathered, coef)
        terms = oracle.pool_gathered(bo, np.abs(gathered), None if coef is None else np.abs(coef))
        got = out[tb % w.B, D_off[t]:D_off[t] + D]
        assert_forward_close(got, ref, terms)
        checked += len(tb)
    return checked


def selected_rows(w, weights_dev, momentum_dev, sel):
    """fp16 weights [len(sel), max D] and momentum of the rows with linear keys sel."""
    hb = np.concatenate([[0], np.cumsum(w.E)])
    W_off = np.concatenate([[0], np.cumsum(w.E * w.D)])
    maxD = int(w.D.max())
    t_sel = np.searchsorted(hb, sel, side="right") - 1
    out = np.zeros((len(sel), maxD), np.float16)
    for j, (k, t) in enumerate(zip(sel, t_sel)):
        D = int(w.D[t])
        s = int(W_off[t] + (int(k) - hb[t]) * D)
        out[j, :D] = weights_dev[s:s + D].cpu().numpy()
    m = momentum_dev[torch.as_tensor(np.asarray(sel, np.int64), device=momentum_dev.device)]
    return out, m.cpu().numpy()


def check_selected_rows(w, sel, w0, m0, w1, m1, inputs=None):
    """Rows sel after one backward (w1, m1; before: w0, m0) against
    oracle.backward_selected: momentum within 1e-5 relative, weights within
    1 fp16 ulp, rows without lookups bit-identical.  Returns the rows'
    lookup counts."""
    idx, off, psw = inputs if inputs is not None else host_inputs(w)
    ws, ms, cnt = oracle.backward_selected(tables(w), w.B, idx, off, w.grad_out.cpu().numpy(),
                                           w.lr, w.eps, sel, w0, m0, psw)
    assert_momentum_close(m1, ms)
    assert_weights_within_ulp(w1, ws)
    free = cnt == 0
    assert np.array_equal(w1[free].view(np.uint16), w0[free].view(np.uint16))
    assert np.array_equal(m1[free].view(np.uint32), m0[free].view(np.uint32))
    return cnt


def assert_f32_forward_close(out, ref, abs_terms, n_max, mean=False):
    """fp32 weights: the kernel's compensated sum is within its final
    rounding plus gamma_{2n}^2 ~ 4 (n u)^2 of the sum of |terms| of the exact
    sum, u = 2^-24, n the bag length (Ogita, Rump and Oishi, Sum2 / Dot2: up
    to two error terms per lookup go to the low part); the oracle's double
    sum, rounded once, within half an ulp.  So |out - ref| <= 1 ulp (2 with
    the mean factor's rounding) + 8 (n u)^2 sum|terms|, about 1e-9 of
    sum|terms| for bags of 200 lookups: a plain fp32 accumulation, off by up
    to about n u of it, would not pass."""
    u = 2.0 ** -24
    ref64 = ref.astype(np.float64)
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    tol = (2 if mean else 1) * ulp + 8 * (n_max * u) ** 2 * abs_terms.astype(np.float64) + 1e-45
    err = np.abs(out.astype(np.float64) - ref64)
    bad = err > tol
    assert not bad.any(), (f"{bad.sum()} of {bad.size} fp32 forward outputs off; worst err "
                           f"{err.max():.3e}, tol there {tol.flat[np.argmax(err - tol)]:.3e}")
    return float(np.max(err / np.maximum(abs_terms.astype(np.float64), 1e-300)))


def assert_f32_step_close(tab, B, indices, offsets, grad_out, psw, mean, lr, eps, w_old, m_old,
                          w_gpu, m_gpu, w_ref, m_ref, elementwise=False):
    """fp32 weights after one Adagrad step against the oracle's (which forms
    the step in fp64 and rounds once).  Each element's gradient g is an fp32
    sum of its row's n terms: within d = (2 n + 10) 2^-24 S of the exact sum,
    S the sum of the terms' magnitudes (as in assert_elementwise_step_close).
    The accumulator (one per row, m = m_old + mean g^2, or one per element)
    is then off by what d moves it plus its fp32 roundings, and the step
    lr g / (sqrt(m) + eps) by what both errors move it plus its own three
    fp32 roundings; the weight may further differ by the rounding of the
    subtraction and one ulp.  Untouched rows must be bit-identical.  Row-wise
    momentum must also be within 1e-5 relative."""
    u = 2.0 ** -24
    ukeys, count, row, flat, col = _touched_elements(tab, B, indices, offsets)
    keys, g = oracle.row_gradients(tab, B, indices, offsets, grad_out, psw, mean)
    absp = None if psw is None else np.abs(psw)
    _, S = oracle.row_gradients(tab, B, indices, offsets, np.abs(grad_out), absp, mean)
    assert np.array_equal(keys.astype(np.int64), ukeys)
    g = g[row, col]
    S = S[row, col]
    d = (2 * count[row] + 10) * u * S
    if elementwise:
        mr = m_ref[flat].astype(np.float64)
        mg = m_gpu[flat].astype(np.float64)
        dm = 4 * u * mr + (2 * np.abs(g) + d) * d
    else:
        Drow = np.asarray(tab.D, np.int64)[np.searchsorted(tab.hash_base, ukeys, side="right") - 1]
        per_row = np.zeros(len(ukeys))
        np.add.at(per_row, row, (2 * np.abs(g) + d) * d)
        mr_row = m_ref[ukeys].astype(np.float64)
        dm_row = 4 * u * mr_row + per_row / Drow
        mg_row = m_gpu[ukeys].astype(np.float64)
        assert np.all(np.abs(mg_row - mr_row) <= dm_row), "row momentum beyond the fp32 bound"
        assert_momentum_close(m_gpu[ukeys], m_ref[ukeys])
        mr, mg, dm = mr_row[row], mg_row[row], dm_row[row]
    assert np.all(np.abs(mg - mr) <= dm), "momentum beyond the fp32 bound"
    wo = np.asarray(w_old, np.float64)[flat]
    wr = np.asarray(w_ref, np.float64)[flat]
    wg = np.asarray(w_gpu, np.float64)[flat]
    lo = np.sqrt(np.maximum(mr - dm, 0.0)) + eps
    hi = np.sqrt(mr + dm) + eps
    step = lr * np.abs(g) / lo
    ds = lr * d / lo + lr * np.abs(g) * (1.0 / lo - 1.0 / hi) + 8 * u * step
    spacing = lambda v: np.spacing(np.abs(v).astype(np.float32)).astype(np.float64)
    tol = ds + 2 * u * (np.abs(wo) + step) + np.maximum(spacing(wr), spacing(wg))
    err = np.abs(wg - wr)
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} of {flat.size} fp32 weights beyond the fp32 bound"
    beyond = int((err > spacing(wr)).sum())
    mask = np.ones(np.asarray(w_gpu).size, bool)
    mask[flat] = False
    assert np.array_equal(np.asarray(w_gpu, np.float32).view(np.uint32)[mask],
                          np.asarray(w_old, np.float32).view(np.uint32)[mask])
    if elementwise:
        assert np.array_equal(np.asarray(m_gpu).view(np.uint32)[mask],
                              np.asarray(m_old, np.float32).view(np.uint32)[mask])
    else:
        free = np.ones(np.asarray(m_gpu).size, bool)
        free[ukeys] = False
        assert np.array_equal(np.asarray(m_gpu).view(np.uint32)[free],
                              np.asarray(m_old, np.float32).view(np.uint32)[free])
    print(f"fp32 step: {flat.size} touched elements, {beyond} beyond 1 ulp of the oracle")
