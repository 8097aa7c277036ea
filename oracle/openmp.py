"""The oracle's forward and backward with their loops spread over the host's
cores (OpenMP) -- TEST INFRASTRUCTURE ONLY: the timed CPU baseline.

Same arguments and results as ``oracle.forward`` and
``oracle.backward_rowwise_adagrad``, bit for bit (tbe_oracle_openmp.cpp forms
every number with the oracle's own helpers, in the oracle's order); the
thread count is OpenMP's (every core unless set_threads or OMP_NUM_THREADS
says otherwise).  Only the
bench's CPU baseline and the tests use it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import Tables, _c, _check, _idx, _p, _weight_bits  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tbe_oracle_openmp.cpp")
_DEPS = (_SRC, os.path.join(_HERE, "tbe_oracle.cpp"))
_LIB = os.path.join(_HERE, "liboracle_openmp.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile with g++ -fopenmp (the oracle's flags otherwise) into
    liboracle_openmp.so."""
    newest = max(os.path.getmtime(f) for f in _DEPS)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
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
        lib.oracle_omp_threads.restype = i32
        lib.oracle_omp_set_threads.argtypes = [i32]
        lib.oracle_omp_forward.argtypes = [i32, i32, P, P, P, P, i32, P, P, i64, P, i32, i32, P]
        lib.oracle_omp_backward.argtypes = [i32, i32, P, P, P, i32, P, P, i64, P, P, i32, i32,
                                            i32, f32, f32, P, P]
        _lib = lib
    return _lib


def threads() -> int:
    """Threads a parallel region of this library uses."""
    return int(_load().oracle_omp_threads())


def set_threads(n: int) -> None:
    """Threads of the parallel regions that follow (OMP_NUM_THREADS is read
    only when the process's OpenMP runtime starts, which importing torch may
    already have done)."""
    _load().oracle_omp_set_threads(int(n))


def forward(tables: Tables, B, weights, indices, offsets, psw=None, mean=False, bf16=False,
            fp32=False):
    """As oracle.forward."""
    lib = _load()
    indices, offsets, bits = _idx(indices, offsets)
    w, wtype = _weight_bits(weights, bf16, fp32)
    psw = _c(psw, np.float32)
    out = np.zeros((B, int(tables.D_offsets[-1])), dtype=np.float32)
    rc = lib.oracle_omp_forward(tables.T, B, _p(tables.D_offsets), _p(tables.hash_base),
                                _p(tables.w_offsets), _p(w), bits, _p(indices), _p(offsets),
                                len(indices), _p(psw), int(bool(mean)), wtype, _p(out))
    _check(rc, "openmp forward")
    return out


def backward_rowwise_adagrad(tables: Tables, B, indices, offsets, grad_out, weights, momentum,
                             lr, eps, psw=None, mean=False, bf16=False, elementwise=False,
                             fp32=False):
    """As oracle.backward_rowwise_adagrad: returns (new_weights, new_momentum)."""
    lib = _load()
    indices, offsets, bits = _idx(indices, offsets)
    w, wtype = _weight_bits(weights, bf16, fp32)
    w = w.copy()
    m = np.array(momentum, dtype=np.float32, copy=True)
    if m.size != (int(tables.w_offsets[-1]) if elementwise else int(tables.hash_base[-1])):
        raise ValueError("momentum has one entry per weight element (elementwise) or per row")
    grad_out = _c(grad_out, np.float32)
    psw = _c(psw, np.float32)
    rc = lib.oracle_omp_backward(tables.T, B, _p(tables.D_offsets), _p(tables.hash_base),
                                 _p(tables.w_offsets), bits, _p(indices), _p(offsets),
                                 len(indices), _p(psw), _p(grad_out), int(bool(mean)), wtype,
                                 int(bool(elementwise)), float(lr), float(eps), _p(w), _p(m))
    _check(rc, "openmp backward")
    return (w.view(np.float16) if wtype == 0 else w), m
