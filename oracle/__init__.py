"""TBE oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow CPU statement of the TBE pooled forward, the sort / run-length
preprocessing and the exact row-wise Adagrad backward, written in C++ with
double accumulation (tbe_oracle.cpp says which passage each function follows).
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline /
reference arm may import this module.  It shares no code with the CUDA library
and never imports it.

All arrays are numpy arrays on the host.  Weights are fp16 (numpy float16),
indices / offsets int32 or int64, per-sample weights and gradients float32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tbe_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (plain -O2, no fast-math) into liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared",
                               "-ffp-contract=off", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_double_to_half.argtypes = [ctypes.c_double]
        lib.oracle_double_to_half.restype = ctypes.c_uint16
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_forward.argtypes = [i32, i32, P, P, P, P, i32, P, P, i64, P, i32, i32, P]
        lib.oracle_pool_gathered.argtypes = [i64, i32, P, P, P, P]
        lib.oracle_preprocess.argtypes = [i32, i32, P, i32, P, P, i64, P, P, P, P, P, P, P]
        lib.oracle_row_gradients.argtypes = [i32, i32, P, P, i32, P, P, i64, P, P, i32, i32, P,
                                             P, P]
        lib.oracle_backward_rowwise_adagrad.argtypes = [i32, i32, P, P, P, i32, P, P, i64, P, P,
                                                        i32, i32, i32, f32, f32, P, P]
        lib.oracle_backward_selected.argtypes = [i32, i32, P, P, i32, P, P, i64, P, P, i32, f32,
                                                 f32, i64, P, i32, P, P, P]
        lib.oracle_repair_offsets.argtypes = [i32, P, i64, i64, P]
        lib.oracle_repair_offsets.restype = i64
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _idx(indices, offsets):
    indices = np.ascontiguousarray(indices)
    offsets = np.ascontiguousarray(offsets)
    if indices.dtype not in (np.int32, np.int64) or offsets.dtype != indices.dtype:
        raise TypeError("indices and offsets must share dtype int32 or int64")
    return indices, offsets, 32 if indices.dtype == np.int32 else 64


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid input (status {rc})")


def bf16_to_double(h: int) -> float:
    return _load().oracle_bf16_to_double(h)


def double_to_bf16(x: float) -> int:
    return _load().oracle_double_to_bf16(x)


def half_to_double(h: int) -> float:
    return _load().oracle_half_to_double(int(h))


def double_to_half(x: float) -> int:
    return int(_load().oracle_double_to_half(float(x)))


class Tables:
    """Table metadata: per-table rows E_t and widths D_t, plus the derived
    cumulative arrays D_offsets, hash_base and weight offsets (int64)."""

    def __init__(self, E, D):
        self.E = np.asarray(E, dtype=np.int64)
        self.D = np.asarray(D, dtype=np.int64)
        self.T = len(self.E)
        self.D_offsets = np.concatenate([[0], np.cumsum(self.D)]).astype(np.int64)
        self.hash_base = np.concatenate([[0], np.cumsum(self.E)]).astype(np.int64)
        self.w_offsets = np.concatenate([[0], np.cumsum(self.E * self.D)]).astype(np.int64)


def _weight_bits(weights, bf16, fp32=False):
    """The weights as the oracle reads them: fp16 values (numpy float16) as
    16-bit patterns; with bf16, bfloat16 bit patterns given as uint16; with
    fp32, float32 values."""
    if bf16 and fp32:
        raise ValueError("one weight type at a time")
    if fp32:
        return np.ascontiguousarray(weights, dtype=np.float32), 2
    if bf16:
        return np.ascontiguousarray(weights, dtype=np.uint16), 1
    return np.ascontiguousarray(weights, dtype=np.float16).view(np.uint16), 0


def forward(tables: Tables, B, weights, indices, offsets, psw=None, mean=False, bf16=False,
            fp32=False):
    """Pooled forward; returns fp32 [B, sum D].  mean: each bag's sum times
    1/L for its L > 1 lookups (HugeCTR's mean combiner).  bf16: weights are
    bfloat16 bit patterns (uint16); fp32: weights are float32."""
    lib = _load()
    indices, offsets, bits = _idx(indices, offsets)
    w, wtype = _weight_bits(weights, bf16, fp32)
    psw = _c(psw, np.float32)
    out = np.zeros((B, int(tables.D_offsets[-1])), dtype=np.float32)
    rc = lib.oracle_forward(tables.T, B, _p(tables.D_offsets), _p(tables.hash_base),
                            _p(tables.w_offsets), _p(w), bits, _p(indices), _p(offsets),
                            len(indices), _p(psw), int(bool(mean)), wtype, _p(out))
    _check(rc, "forward")
    return out


def pool_gathered(bag_off, rows, coef=None):
    """Pool pre-gathered fp16 rows [nlookups, D] into bags given by bag_off."""
    lib = _load()
    bag_off = _c(bag_off, np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.float16)
    D = rows.shape[1]
    coef = _c(coef, np.float32)
    out = np.zeros((len(bag_off) - 1, D), dtype=np.float32)
    rc = lib.oracle_pool_gathered(len(bag_off) - 1, D, _p(bag_off), _p(rows.view(np.uint16)),
                                  _p(coef), _p(out))
    _check(rc, "pool_gathered")
    return out


def preprocess(tables: Tables, B, indices, offsets):
    """Returns dict(sorted_keys, sorted_bags, sorted_pos, unique_keys, run_starts)."""
    lib = _load()
    indices, offsets, bits = _idx(indices, offsets)
    n = len(indices)
    sk = np.zeros(n, np.uint32)
    sb = np.zeros(n, np.uint32)
    sp = np.zeros(n, np.int64)
    uk = np.zeros(n, np.uint32)
    rs = np.zeros(n + 1, np.int64)
    nv = np.zeros(1, np.int64)
    R = np.zeros(1, np.int64)
    rc = lib.oracle_preprocess(tables.T, B, _p(tables.hash_base), bits, _p(indices), _p(offsets),
                               n, _p(sk), _p(sb), _p(sp), _p(uk), _p(rs), _p(nv), _p(R))
    _check(rc, "preprocess")
    nv, R = int(nv[0]), int(R[0])
    return dict(sorted_keys=sk[:nv], sorted_bags=sb[:nv], sorted_pos=sp[:nv],
                unique_keys=uk[:R], run_starts=rs[:R + 1])


def row_gradients(tables: Tables, B, indices, offsets, grad_out, psw=None, mean=False):
    """Summed gradient (double) of every touched row: (keys[R], g[R, maxD]).
    mean: each bag's gradient times 1/L for its L > 1 lookups, before grouping."""
    lib = _load()
    indices, offsets, bits = _idx(indices, offsets)
    n = len(indices)
    maxD = int(tables.D.max())
    keys = np.zeros(max(n, 1), np.uint32)
    g = np.zeros((max(n, 1), maxD), np.float64)
    R = np.zeros(1, np.int64)
    grad_out = _c(grad_out, np.float32)
    psw = _c(psw, np.float32)
    rc = lib.oracle_row_gradients(tables.T, B, _p(tables.D_offsets), _p(tables.hash_base), bits,
                                  _p(indices), _p(offsets), n, _p(psw), _p(grad_out),
                                  int(bool(mean)), maxD, _p(keys), _p(g), _p(R))
    _check(rc, "row_gradients")
    R = int(R[0])
    return keys[:R], g[:R]


def backward_rowwise_adagrad(tables: Tables, B, indices, offsets, grad_out, weights, momentum,
                             lr, eps, psw=None, mean=False, bf16=False, elementwise=False,
                             fp32=False):
    """Returns (new_weights, new_momentum fp32); inputs are not modified.
    mean: each bag's gradient times 1/L for its L > 1 lookups, before grouping.
    bf16: weights (in and out) are bfloat16 bit patterns (uint16); fp32:
    float32 weights; else fp16.
    elementwise: HugeCTR's element-wise Adagrad, momentum shaped like the
    flat weights (one accumulator per element), instead of one per row."""
    lib = _load()
    indices, offsets, bits = _idx(indices, offsets)
    w, wtype = _weight_bits(weights, bf16, fp32)
    w = w.copy()
    m = np.array(momentum, dtype=np.float32, copy=True)
    if m.size != (int(tables.w_offsets[-1]) if elementwise else int(tables.hash_base[-1])):
        raise ValueError("momentum has one entry per weight element (elementwise) or per row")
    grad_out = _c(grad_out, np.float32)
    psw = _c(psw, np.float32)
    rc = lib.oracle_backward_rowwise_adagrad(tables.T, B, _p(tables.D_offsets),
                                             _p(tables.hash_base), _p(tables.w_offsets), bits,
                                             _p(indices), _p(offsets), len(indices), _p(psw),
                                             _p(grad_out), int(bool(mean)), wtype,
                                             int(bool(elementwise)), float(lr), float(eps),
                                             _p(w), _p(m))
    _check(rc, "backward")
    return (w.view(np.float16) if wtype == 0 else w), m


def backward_selected(tables: Tables, B, indices, offsets, grad_out, lr, eps, sel_keys, w_rows,
                      m_rows, psw=None, mean=False):
    """Row-wise Adagrad for selected linear keys only.

    w_rows [nsel, maxD] fp16 and m_rows [nsel] fp32 hold the rows' values before
    the step; returns (w_rows_new, m_rows_new, run_lengths)."""
    lib = _load()
    indices, offsets, bits = _idx(indices, offsets)
    sel = _c(sel_keys, np.uint32)
    maxD = int(tables.D.max())
    w = np.array(w_rows, dtype=np.float16, copy=True).reshape(len(sel), maxD)
    m = np.array(m_rows, dtype=np.float32, copy=True)
    cnt = np.zeros(len(sel), np.int64)
    grad_out = _c(grad_out, np.float32)
    psw = _c(psw, np.float32)
    rc = lib.oracle_backward_selected(tables.T, B, _p(tables.D_offsets), _p(tables.hash_base),
                                      bits, _p(indices), _p(offsets), len(indices), _p(psw),
                                      _p(grad_out), int(bool(mean)), float(lr), float(eps),
                                      len(sel), _p(sel),
                                      maxD, _p(w.view(np.uint16)), _p(m), _p(cnt))
    _check(rc, "backward_selected")
    return w, m, cnt


def repair_offsets(offsets, n):
    """Offset repair reading: returns (repaired int64 offsets, number changed)."""
    lib = _load()
    offsets = np.ascontiguousarray(offsets)
    bits = 32 if offsets.dtype == np.int32 else 64
    out = np.zeros(len(offsets), np.int64)
    changed = lib.oracle_repair_offsets(bits, _p(offsets), len(offsets), int(n), _p(out))
    return out, int(changed)
