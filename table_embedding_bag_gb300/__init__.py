"""Thin Python binding of libtbe.so, the GB300 Table Batched Embedding library.

Every function here only marshals arguments (device pointers from torch
tensors, the current CUDA stream) into the C ABI declared in include/tbe.h;
every step of the computation runs in the library's CUDA kernels.  There is
no CPU fallback: if libtbe.so is missing or fails to load, the functions
raise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import _build

__all__ = [
    "build", "TBEDesc", "Workspace", "TBEError", "tbe_workspace_size", "tbe_forward",
    "tbe_preprocess", "tbe_backward_rowwise_adagrad", "tbe_workspace_view", "tbe_read_status",
    "tbe_version", "tbe_kernel_launches", "tbe_probe_set", "tbe_probe_read",
    "TableBatchedEmbedding", "lib_path", "tbe_backward_rowwise_adagrad_noalloc",
    "TBE_NOALLOC_SCRATCH_BYTES", "TBE_ETOO_LARGE",
    "TBE_F_CHECK_BOUNDS", "TBE_F_REPAIR_OFFSETS", "TBE_F_FORCE_GENERIC", "TBE_F_LONG_TWO_LAUNCH",
    "TBE_F_PREPROCESSED", "TBE_F_MEAN", "TBE_F_ELEMENTWISE", "TBE_WS_WEIGHTED", "TBE_WS_MEAN", "TBE_ERR_INDEX_RANGE", "TBE_ERR_OFFSETS",
]

TBE_OK, TBE_EINVAL, TBE_EWORKSPACE, TBE_EUNSUPPORTED, TBE_ECUDA, TBE_ETOO_LARGE = range(6)
TBE_NOALLOC_SCRATCH_BYTES = 32 << 20
TBE_DT_F16, TBE_DT_I32, TBE_DT_I64, TBE_DT_BF16, TBE_DT_F32 = 1, 2, 3, 4, 5
TBE_F_CHECK_BOUNDS = 1 << 0
TBE_F_REPAIR_OFFSETS = 1 << 1
TBE_F_FORCE_GENERIC = 1 << 2
TBE_F_LONG_TWO_LAUNCH = 1 << 3
TBE_F_PREPROCESSED = 1 << 4
TBE_F_MEAN = 1 << 5
TBE_F_ELEMENTWISE = 1 << 6
TBE_WS_MEAN = 1 << 1
TBE_WS_WEIGHTED = 1 << 0
TBE_ERR_INDEX_RANGE = 1 << 0
TBE_ERR_OFFSETS = 1 << 1
TBE_ERR_TIMEOUT = 1 << 2
# kernels tbe_probe_set can time
TBE_PROBE_OFF = 0
TBE_PROBE_EXPAND_COUNT = 1
TBE_PROBE_RADIX_DOWNSWEEP = 2
TBE_PROBE_FORWARD_HOT = 3
TBE_PROBE_FORWARD_COLD = 4
TBE_PROBE_SHORT_RUNS = 5
TBE_PROBE_MEDIUM_RUNS = 6
TBE_PROBE_LONG_CHUNKS = 7
TBE_PROBE_HOT_GRAD = 8
_STATUS_NAMES = {1: "TBE_EINVAL", 2: "TBE_EWORKSPACE", 3: "TBE_EUNSUPPORTED", 4: "TBE_ECUDA",
                 5: "TBE_ETOO_LARGE"}

lib_path = _build.LIB
build = _build.build


class TBEError(RuntimeError):
    def __init__(self, call, code):
        super().__init__(f"{call} failed: {_STATUS_NAMES.get(code, code)}")
        self.code = code


class tbe_desc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("B", ctypes.c_int32),
                ("weights_dtype", ctypes.c_int32), ("index_dtype", ctypes.c_int32),
                ("D_offsets", ctypes.c_void_p), ("hash_base", ctypes.c_void_p),
                ("weights_offsets", ctypes.c_void_p), ("total_D", ctypes.c_int64),
                ("total_E", ctypes.c_int64), ("max_D", ctypes.c_int32),
                ("min_D", ctypes.c_int32)]


class tbe_ws_view(ctypes.Structure):
    _fields_ = [("sorted_keys", ctypes.c_void_p), ("sorted_bags", ctypes.c_void_p),
                ("sorted_psw", ctypes.c_void_p), ("unique_keys", ctypes.c_void_p),
                ("run_starts", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("long_runs", ctypes.c_void_p), ("long_threshold", ctypes.c_int32),
                ("chunk", ctypes.c_int32), ("run_pairs", ctypes.c_void_p),
                ("pair_starts", ctypes.c_void_p), ("pair_bags", ctypes.c_void_p),
                ("hot_keys", ctypes.c_void_p), ("hot_n", ctypes.c_void_p),
                ("hot_slots", ctypes.c_int32), ("medium_threshold", ctypes.c_int32)]


_lib = None


def configure(lib):
    """Declare the C signatures of the entry points on a loaded libtbe (a
    ctypes.CDLL); returns lib."""
    P, i64, u32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32,
                            ctypes.c_float, ctypes.c_size_t)
    D = ctypes.POINTER(tbe_desc)
    lib.tbe_workspace_size.argtypes = [D, i64, u32, ctypes.POINTER(sz)]
    lib.tbe_forward.argtypes = [D, P, P, P, i64, P, P, P, sz, P, u32]
    lib.tbe_preprocess.argtypes = [D, P, P, i64, P, P, sz, P, u32]
    lib.tbe_backward_rowwise_adagrad.argtypes = [D, P, P, P, i64, P, P, P, f32, f32, P, sz, P,
                                                 u32]
    lib.tbe_workspace_view.argtypes = [D, i64, u32, P, ctypes.POINTER(tbe_ws_view)]
    lib.tbe_backward_rowwise_adagrad_noalloc.argtypes = [D, P, P, P, i64, P, P, P, f32, f32,
                                                         P, u32]
    lib.tbe_read_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
    lib.tbe_version.restype = ctypes.c_char_p
    lib.tbe_kernel_launches.restype = ctypes.c_uint64
    lib.tbe_kernel_launches.argtypes = []
    lib.tbe_probe_set.argtypes = [u32]
    lib.tbe_probe_read.argtypes = [ctypes.POINTER(ctypes.c_uint32),
                                   ctypes.POINTER(ctypes.c_float)]
    for f in ("tbe_workspace_size", "tbe_forward", "tbe_preprocess",
              "tbe_backward_rowwise_adagrad", "tbe_workspace_view", "tbe_read_status",
              "tbe_backward_rowwise_adagrad_noalloc", "tbe_probe_set", "tbe_probe_read"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(lib_path):
            raise RuntimeError(f"{lib_path} is not built; run table_embedding_bag_gb300.build()")
        _lib = configure(ctypes.CDLL(lib_path))
    return _lib


def _ok(call, code):
    if code != TBE_OK:
        raise TBEError(call, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


_WEIGHT_DT = {torch.float16: TBE_DT_F16, torch.bfloat16: TBE_DT_BF16,
              torch.float32: TBE_DT_F32}


class TBEDesc:
    """Problem description: per-table rows E_t and widths D_t, bags per table B,
    index dtype and weight dtype (torch.float16, torch.bfloat16 or torch.float32).  Holds the
    three cumulative int64 arrays on the device."""

    def __init__(self, E, D, B, index_dtype=torch.int64, device="cuda",
                 weights_dtype=torch.float16):
        self.E = np.asarray(E, dtype=np.int64)
        self.D = np.asarray(D, dtype=np.int64)
        if self.E.ndim != 1 or self.E.shape != self.D.shape or len(self.E) == 0:
            raise ValueError("E and D must be equal-length 1-d sequences")
        if np.any(self.D % 8) or np.any(self.D < 8) or np.any(self.D > 1024):
            raise ValueError("every D_t must be a multiple of 8 in [8, 1024]")
        self.T, self.B = len(self.E), int(B)
        self.index_dtype = index_dtype
        if weights_dtype not in _WEIGHT_DT:
            raise ValueError("weights_dtype must be torch.float16, torch.bfloat16 or "
                             "torch.float32")
        self.weights_dtype = weights_dtype
        cum = lambda a: np.concatenate([[0], np.cumsum(a)]).astype(np.int64)
        self.D_offsets_h = cum(self.D)
        self.hash_base_h = cum(self.E)
        self.weights_offsets_h = cum(self.E * self.D)
        dev = torch.device(device)
        self.D_offsets = torch.from_numpy(self.D_offsets_h).to(dev)
        self.hash_base = torch.from_numpy(self.hash_base_h).to(dev)
        self.weights_offsets = torch.from_numpy(self.weights_offsets_h).to(dev)
        self.total_D = int(self.D_offsets_h[-1])
        self.total_E = int(self.hash_base_h[-1])
        self.num_weights = int(self.weights_offsets_h[-1])
        self.c = tbe_desc(self.T, self.B, _WEIGHT_DT[weights_dtype],
                          TBE_DT_I32 if index_dtype == torch.int32 else TBE_DT_I64,
                          self.D_offsets.data_ptr(), self.hash_base.data_ptr(),
                          self.weights_offsets.data_ptr(), self.total_D, self.total_E,
                          int(self.D.max()), int(self.D.min()))

    @property
    def ref(self):
        return ctypes.byref(self.c)


def tbe_workspace_size(desc: TBEDesc, n_max: int, weighted: bool = False,
                       mean: bool = False) -> int:
    out = ctypes.c_size_t(0)
    ws_flags = (TBE_WS_WEIGHTED if weighted else 0) | (TBE_WS_MEAN if mean else 0)
    _ok("tbe_workspace_size", _load().tbe_workspace_size(
        desc.ref, int(n_max), ws_flags, ctypes.byref(out)))
    return out.value


class Workspace:
    """Device workspace for calls with at most n_max lookups."""

    def __init__(self, desc: TBEDesc, n_max: int, weighted: bool = False, device="cuda",
                 mean: bool = False):
        self.nbytes = tbe_workspace_size(desc, n_max, weighted, mean)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)
        self.weighted = weighted

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())


def _check_tensors(desc, indices, offsets):
    if indices.dtype != desc.index_dtype or offsets.dtype != desc.index_dtype:
        raise TypeError(f"indices and offsets must be {desc.index_dtype}")
    if offsets.numel() != desc.T * desc.B + 1:
        raise ValueError("offsets must have T*B+1 entries")
    if not (indices.is_contiguous() and offsets.is_contiguous()):
        raise ValueError("indices and offsets must be contiguous")


def _check_weights(desc, weights):
    if isinstance(weights, torch.Tensor):
        if weights.dtype != desc.weights_dtype:
            raise TypeError(f"weights must be {desc.weights_dtype}")
        if weights.numel() < desc.num_weights:
            raise ValueError(f"weights must hold {desc.num_weights} elements")


def _check_dense(desc, t, name):
    """out / grad_out: fp32, contiguous, B x total_D elements."""
    if isinstance(t, torch.Tensor):
        if t.dtype != torch.float32 or not t.is_contiguous() or \
                t.numel() != desc.B * desc.total_D:
            raise ValueError(f"{name} must be contiguous float32 [{desc.B}, {desc.total_D}]")


def _check_psw(indices, psw):
    if isinstance(psw, torch.Tensor):
        if psw.dtype != torch.float32 or not psw.is_contiguous() or \
                psw.numel() != indices.numel():
            raise ValueError("per_sample_weights must be contiguous float32, one per lookup")


def _check_momentum(desc, momentum, flags):
    """The accumulators the update writes: one per row, or one per weight
    element with TBE_F_ELEMENTWISE."""
    if isinstance(momentum, torch.Tensor):
        need = desc.num_weights if flags & TBE_F_ELEMENTWISE else desc.total_E
        if momentum.dtype != torch.float32 or momentum.numel() < need:
            raise ValueError(f"momentum must be float32 with {need} entries")


def tbe_forward(desc: TBEDesc, weights, indices, offsets, per_sample_weights, out, ws: Workspace,
                flags: int = 0, stream=None):
    """Pooled forward into out (fp32 [B, sum D]); see tbe_forward in include/tbe.h."""
    _check_tensors(desc, indices, offsets)
    _check_weights(desc, weights)
    _check_dense(desc, out, "out")
    _check_psw(indices, per_sample_weights)
    _ok("tbe_forward", _load().tbe_forward(
        desc.ref, _ptr(weights), _ptr(indices), _ptr(offsets), indices.numel(),
        _ptr(per_sample_weights), _ptr(out), ws.ptr, ws.nbytes, _stream(stream), flags))
    return out


def tbe_preprocess(desc: TBEDesc, indices, offsets, per_sample_weights, ws: Workspace,
                   flags: int = 0, stream=None):
    _check_tensors(desc, indices, offsets)
    _check_psw(indices, per_sample_weights)
    _ok("tbe_preprocess", _load().tbe_preprocess(
        desc.ref, _ptr(indices), _ptr(offsets), indices.numel(), _ptr(per_sample_weights),
        ws.ptr, ws.nbytes, _stream(stream), flags))


def tbe_backward_rowwise_adagrad(desc: TBEDesc, grad_out, indices, offsets, per_sample_weights,
                                 weights, momentum, lr, eps, ws: Workspace, flags: int = 0,
                                 stream=None):
    """Backward with one Adagrad update per touched row (row-wise, or
    element-wise with TBE_F_ELEMENTWISE), in place on weights and momentum;
    see include/tbe.h."""
    _check_tensors(desc, indices, offsets)
    _check_weights(desc, weights)
    _check_momentum(desc, momentum, flags)
    _check_dense(desc, grad_out, "grad_out")
    _check_psw(indices, per_sample_weights)
    _ok("tbe_backward_rowwise_adagrad", _load().tbe_backward_rowwise_adagrad(
        desc.ref, _ptr(grad_out), _ptr(indices), _ptr(offsets), indices.numel(),
        _ptr(per_sample_weights), _ptr(weights), _ptr(momentum), float(lr), float(eps), ws.ptr,
        ws.nbytes, _stream(stream), flags))


def tbe_backward_rowwise_adagrad_noalloc(desc: TBEDesc, grad_out, indices, offsets,
                                         per_sample_weights, weights, momentum, lr, eps,
                                         flags: int = 0, stream=None):
    """The backward without any workspace: for callers that must not allocate
    device memory at call time (see tbe_backward_rowwise_adagrad_noalloc in
    include/tbe.h for the scratch limit and the rules on overlapping calls)."""
    _check_tensors(desc, indices, offsets)
    _check_weights(desc, weights)
    _check_momentum(desc, momentum, flags)
    _check_dense(desc, grad_out, "grad_out")
    _check_psw(indices, per_sample_weights)
    _ok("tbe_backward_rowwise_adagrad_noalloc", _load().tbe_backward_rowwise_adagrad_noalloc(
        desc.ref, _ptr(grad_out), _ptr(indices), _ptr(offsets), indices.numel(),
        _ptr(per_sample_weights), _ptr(weights), _ptr(momentum), float(lr), float(eps),
        _stream(stream), flags))


def tbe_workspace_view(desc: TBEDesc, n: int, ws: Workspace) -> dict:
    """Device pointers into the workspace (sorted keys, runs, ...) as ints."""
    v = tbe_ws_view()
    _ok("tbe_workspace_view", _load().tbe_workspace_view(
        desc.ref, int(n), TBE_WS_WEIGHTED if ws.weighted else 0, ws.ptr, ctypes.byref(v)))
    return {name: getattr(v, name) for name, _ in tbe_ws_view._fields_}


def tbe_read_status(ws: Workspace, stream=None) -> int:
    """Read and clear the device status word (synchronises the stream)."""
    v = ctypes.c_int32(0)
    _ok("tbe_read_status", _load().tbe_read_status(ws.ptr, _stream(stream), ctypes.byref(v)))
    return v.value


def tbe_version() -> str:
    return _load().tbe_version().decode()


def tbe_kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(_load().tbe_kernel_launches())


def tbe_probe_set(kernel: int) -> None:
    """Time every following launch of one kernel (TBE_PROBE_*) with CUDA events."""
    _ok("tbe_probe_set", _load().tbe_probe_set(kernel))


def tbe_probe_read():
    """(launches, total milliseconds) recorded since tbe_probe_set; waits for the events."""
    n = ctypes.c_uint32(0)
    ms = ctypes.c_float(0.0)
    _ok("tbe_probe_read", _load().tbe_probe_read(ctypes.byref(n), ctypes.byref(ms)))
    return int(n.value), float(ms.value)


class TableBatchedEmbedding:
    """Owns 16-bit weights (fp16, or bf16), fp32 Adagrad momentum (one value
    per row, or per weight element with elementwise=True) and a workspace for
    one problem shape; forward() and backward() call the C ABI, with mean
    pooling throughout when mean=True."""

    def __init__(self, E, D, B, n_max, index_dtype=torch.int64, weighted=False, weights=None,
                 momentum=None, lr=0.01, eps=1e-8, device="cuda", weights_dtype=torch.float16,
                 elementwise=False, mean=False):
        self.desc = TBEDesc(E, D, B, index_dtype, device, weights_dtype)
        self.ws = Workspace(self.desc, n_max, weighted, device, mean=mean)
        self.mean = mean
        self.weights = weights if weights is not None else torch.zeros(
            self.desc.num_weights, dtype=weights_dtype, device=device)
        self.elementwise = elementwise
        n_mom = self.desc.num_weights if elementwise else self.desc.total_E
        self.momentum = momentum if momentum is not None else torch.zeros(
            n_mom, dtype=torch.float32, device=device)
        if self.momentum.numel() != n_mom:
            raise ValueError(f"momentum must have {n_mom} entries")
        self.lr, self.eps = lr, eps
        self.out = torch.empty(self.desc.B, self.desc.total_D, dtype=torch.float32, device=device)

    def forward(self, indices, offsets, per_sample_weights=None, flags=0):
        return tbe_forward(self.desc, self.weights, indices, offsets, per_sample_weights,
                           self.out, self.ws, flags | (TBE_F_MEAN if self.mean else 0))

    def backward(self, grad_out, indices, offsets, per_sample_weights=None, flags=0):
        tbe_backward_rowwise_adagrad(self.desc, grad_out, indices, offsets, per_sample_weights,
                                     self.weights, self.momentum, self.lr, self.eps, self.ws,
                                     flags | (TBE_F_ELEMENTWISE if self.elementwise else 0) |
                                     (TBE_F_MEAN if self.mean else 0))
