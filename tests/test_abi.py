"""The C-ABI library builds, loads without a GPU, exports every function that
include/tbe.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest
import torch

import table_embedding_bag_gb300 as tbe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    tbe.build()
    return ctypes.CDLL(tbe.lib_path)


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tbe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tbe_[a-z_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted([
        "tbe_backward_rowwise_adagrad", "tbe_backward_rowwise_adagrad_noalloc", "tbe_forward",
        "tbe_preprocess", "tbe_read_status", "tbe_version", "tbe_workspace_size",
        "tbe_kernel_launches", "tbe_probe_set", "tbe_probe_read",
        "tbe_workspace_view"])


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_string(lib):
    lib.tbe_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.tbe_version()


def _desc(T=2, B=4, E=(10, 20), D=(8, 16), index=tbe.TBE_DT_I64):
    fake = 0x1000  # never dereferenced by the host-side checks
    return tbe.tbe_desc(T, B, tbe.TBE_DT_F16, index, fake, fake, fake, sum(D), sum(E), max(D),
                        min(D))


def _ws_size(lib, d, n, flags=0):
    out = ctypes.c_size_t(0)
    lib.tbe_workspace_size.argtypes = [ctypes.POINTER(tbe.tbe_desc), ctypes.c_int64,
                                       ctypes.c_uint32, ctypes.POINTER(ctypes.c_size_t)]
    rc = lib.tbe_workspace_size(ctypes.byref(d), n, flags, ctypes.byref(out))
    return rc, out.value


def test_workspace_size_grows_with_lookups_and_weights(lib):
    d = _desc()
    rc0, s0 = _ws_size(lib, d, 0)
    rc1, s1 = _ws_size(lib, d, 1 << 20)
    rc2, s2 = _ws_size(lib, d, 1 << 20, tbe.TBE_WS_WEIGHTED)
    assert rc0 == rc1 == rc2 == tbe.TBE_OK
    assert 0 < s0 < s1 < s2
    assert s2 - s1 >= 2 * 4 * (1 << 20)  # two per-sample-weight buffers


@pytest.mark.parametrize("field,value,code", [
    ("T", 0, tbe.TBE_EINVAL), ("B", 0, tbe.TBE_EINVAL), ("weights_dtype", 9, tbe.TBE_EUNSUPPORTED),
    ("index_dtype", 9, tbe.TBE_EUNSUPPORTED), ("max_D", 2048, tbe.TBE_EUNSUPPORTED),
    ("min_D", 4, tbe.TBE_EUNSUPPORTED), ("total_E", 1 << 32, tbe.TBE_EUNSUPPORTED),
    ("D_offsets", None, tbe.TBE_EINVAL)])
def test_bad_descriptors_rejected(lib, field, value, code):
    d = _desc()
    setattr(d, field, value)
    assert _ws_size(lib, d, 100)[0] == code


def test_bf16_weights_take_the_same_layout_as_fp16(lib):
    # bf16 tables have hot rows too: the same workspace as fp16 tables
    d16, dbf = _desc(B=4096), _desc(B=4096)
    dbf.weights_dtype = tbe.TBE_DT_BF16
    rc16, s16 = _ws_size(lib, d16, 1 << 16)
    rcbf, sbf = _ws_size(lib, dbf, 1 << 16)
    assert rc16 == rcbf == tbe.TBE_OK
    assert sbf == s16


def test_fp32_weights_accepted_without_hot_row_buffers(lib):
    # fp32 tables take the gather paths: no hot-row histograms are laid out
    d16, d32 = _desc(B=4096), _desc(B=4096)
    d32.weights_dtype = tbe.TBE_DT_F32
    rc16, s16 = _ws_size(lib, d16, 1 << 16)
    rc32, s32 = _ws_size(lib, d32, 1 << 16)
    assert rc16 == rc32 == tbe.TBE_OK
    assert s32 < s16


def test_binding_checks_the_weight_dtype():
    with pytest.raises(ValueError):
        tbe.TBEDesc([10], [8], 2, device="cpu", weights_dtype=torch.float64)
    d32 = tbe.TBEDesc([10], [8], 2, device="cpu", weights_dtype=torch.float32)
    assert d32.c.weights_dtype == tbe.TBE_DT_F32
    desc = tbe.TBEDesc([10], [8], 2, device="cpu", weights_dtype=torch.bfloat16)
    idx = torch.zeros(3, dtype=torch.int64)
    off = torch.tensor([0, 1, 3], dtype=torch.int64)
    out = torch.empty(2, 8)
    with pytest.raises(TypeError):  # fp16 weights for a bf16 problem, refused before any call
        tbe.tbe_forward(desc, torch.zeros(80, dtype=torch.float16), idx, off, None, out, None)


def test_bad_sizes_rejected(lib):
    assert _ws_size(lib, _desc(), -1)[0] == tbe.TBE_EINVAL
    assert _ws_size(lib, _desc(), 1 << 33)[0] == tbe.TBE_EUNSUPPORTED


def test_small_workspace_rejected_before_any_launch(lib):
    lib.tbe_kernel_launches.restype = ctypes.c_uint64
    launches0 = lib.tbe_kernel_launches()
    d = _desc()
    P = ctypes.c_void_p
    lib.tbe_forward.argtypes = [ctypes.POINTER(tbe.tbe_desc), P, P, P, ctypes.c_int64, P, P, P,
                                ctypes.c_size_t, P, ctypes.c_uint32]
    fake = P(0x1000)
    rc = lib.tbe_forward(ctypes.byref(d), fake, fake, fake, 10, None, fake, fake, 16, None, 0)
    assert rc == tbe.TBE_EWORKSPACE
    rc = lib.tbe_forward(ctypes.byref(d), fake, fake, fake, 10, None, fake, None, 1 << 30, None, 0)
    assert rc == tbe.TBE_EWORKSPACE
    rc = lib.tbe_forward(ctypes.byref(d), fake, fake, None, 10, None, fake, fake, 1 << 30, None, 0)
    assert rc == tbe.TBE_EINVAL
    lib.tbe_backward_rowwise_adagrad.argtypes = [
        ctypes.POINTER(tbe.tbe_desc), P, P, P, ctypes.c_int64, P, P, P, ctypes.c_float,
        ctypes.c_float, P, ctypes.c_size_t, P, ctypes.c_uint32]
    rc = lib.tbe_backward_rowwise_adagrad(ctypes.byref(d), fake, fake, fake, 10, None, fake, fake,
                                          0.01, 1e-8, fake, 8, None, 0)
    assert rc == tbe.TBE_EWORKSPACE
    assert lib.tbe_kernel_launches() == launches0  # rejected calls launch nothing


def test_package_refuses_to_run_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(tbe, "lib_path", str(tmp_path / "missing.so"))
    monkeypatch.setattr(tbe, "_lib", None)
    with pytest.raises(RuntimeError):
        tbe.tbe_version()


def test_probe_selection_and_empty_record(lib):
    # no GPU needed: selecting a kernel records nothing until it launches
    assert lib.tbe_probe_set(99) == tbe.TBE_EINVAL
    assert lib.tbe_probe_set(tbe.TBE_PROBE_LONG_CHUNKS) == tbe.TBE_OK
    assert tbe.tbe_probe_read() == (0, 0.0)
    assert lib.tbe_probe_set(tbe.TBE_PROBE_OFF) == tbe.TBE_OK


def test_binding_constants_match_the_header():
    import re
    text = open(os.path.join(ROOT, "include", "tbe.h")).read()
    defs = dict(re.findall(r"#define (TBE_(?:F|WS|ERR)_\w+) \((1u? << \d+)\)", text))
    assert defs, "no flag definitions found"
    for name, expr in defs.items():
        assert getattr(tbe, name) == eval(expr.replace("1u", "1")), name
    enum = re.search(r"enum \{ (TBE_DT_[^}]*)\}", text).group(1)
    for name, val in re.findall(r"(TBE_DT_\w+) = (\d+)", enum):
        assert getattr(tbe, name) == int(val), name


def test_module_sizes_state_and_passes_its_flags(monkeypatch):
    # built on the host (no device memory needed); the C calls are captured
    emb = tbe.TableBatchedEmbedding([10, 4], [8, 16], 3, 64, device="cpu",
                                    weights_dtype=torch.bfloat16, elementwise=True, mean=True)
    assert emb.weights.dtype == torch.bfloat16 and emb.weights.numel() == 10 * 8 + 4 * 16
    assert emb.momentum.numel() == emb.weights.numel()  # one accumulator per element
    assert emb.ws.nbytes == tbe.tbe_workspace_size(emb.desc, 64, mean=True)
    assert tbe.TableBatchedEmbedding([10, 4], [8, 16], 3, 64, device="cpu").momentum.numel() == 14
    with pytest.raises(ValueError):
        tbe.TableBatchedEmbedding([10], [8], 3, 64, device="cpu", elementwise=True,
                                  momentum=torch.zeros(10))
    seen = {}
    monkeypatch.setattr(tbe, "tbe_forward", lambda *a: seen.setdefault("fwd", a[-1]))
    monkeypatch.setattr(tbe, "tbe_backward_rowwise_adagrad",
                        lambda *a: seen.setdefault("bwd", a[-1]))
    idx = torch.zeros(2, dtype=torch.int64)
    off = torch.tensor([0, 1, 1, 1, 2, 2, 2], dtype=torch.int64)
    emb.forward(idx, off)
    emb.backward(torch.zeros(3, 24), idx, off, flags=tbe.TBE_F_PREPROCESSED)
    assert seen["fwd"] == tbe.TBE_F_MEAN
    assert seen["bwd"] == tbe.TBE_F_PREPROCESSED | tbe.TBE_F_ELEMENTWISE | tbe.TBE_F_MEAN


@pytest.mark.parametrize("dims", [dict(T=2, B=4, E=(10, 20), D=(8, 16)),
                                  dict(T=3, B=4096, E=(1000, 5, 70000), D=(128, 8, 1024))])
def test_workspace_layout_invariants(lib, dims):
    # Host arithmetic only (a fake base address, nothing dereferenced): every
    # region lies inside the reported size at 256-byte alignment; the hot-row
    # state sits at offsets that depend on the tables alone, so one workspace
    # serves calls of any n, weighted or not, with or without mean pooling;
    # the mean region is the last one.
    d = _desc(**dims)
    base = 1 << 40
    lib.tbe_workspace_view.argtypes = [ctypes.POINTER(tbe.tbe_desc), ctypes.c_int64,
                                       ctypes.c_uint32, ctypes.c_void_p,
                                       ctypes.POINTER(tbe.tbe_ws_view)]
    state = None
    for n in (0, 1000, 1 << 20):
        sizes = {}
        for flags in (0, tbe.TBE_WS_WEIGHTED, tbe.TBE_WS_MEAN,
                      tbe.TBE_WS_WEIGHTED | tbe.TBE_WS_MEAN):
            rc, size = _ws_size(lib, d, n, flags)
            assert rc == tbe.TBE_OK
            sizes[flags] = size
            v = tbe.tbe_ws_view()
            assert lib.tbe_workspace_view(ctypes.byref(d), n, flags, base,
                                          ctypes.byref(v)) == tbe.TBE_OK
            ptrs = {name: getattr(v, name) for name, t in tbe.tbe_ws_view._fields_
                    if t is ctypes.c_void_p and getattr(v, name)}
            for name, p in ptrs.items():
                assert base <= p < base + size, name
                assert (p - base) % 256 == 0, name
            assert ("sorted_psw" in ptrs) == bool(flags & tbe.TBE_WS_WEIGHTED)
            here = (v.hot_keys, v.hot_n, v.counts)
            state = state or here
            assert here == state
        grad = ((4 * dims["B"] * sum(dims["D"]) + 255) // 256) * 256
        assert sizes[tbe.TBE_WS_MEAN] - sizes[0] == grad
        assert sizes[tbe.TBE_WS_WEIGHTED | tbe.TBE_WS_MEAN] - sizes[tbe.TBE_WS_WEIGHTED] == grad


def test_binding_checks_state_sizes_before_any_call():
    # a row-sized accumulator with the element-wise flag (or short weights)
    # would be written past its end: refused on the host
    desc = tbe.TBEDesc([10, 4], [8, 16], 2, device="cpu")
    idx = torch.zeros(1, dtype=torch.int64)
    off = torch.tensor([0, 1, 1, 1, 1], dtype=torch.int64)
    W = torch.zeros(desc.num_weights, dtype=torch.float16)
    G = torch.zeros(2, 24)
    rows, elems = torch.zeros(desc.total_E), torch.zeros(desc.num_weights)
    for fn, extra in ((tbe.tbe_backward_rowwise_adagrad, (None,)),
                      (tbe.tbe_backward_rowwise_adagrad_noalloc, ())):
        with pytest.raises(ValueError):
            fn(desc, G, idx, off, None, W, rows, 0.1, 1e-8, *extra, flags=tbe.TBE_F_ELEMENTWISE)
        with pytest.raises(ValueError):
            fn(desc, G, idx, off, None, W[:-1], elems, 0.1, 1e-8, *extra,
               flags=tbe.TBE_F_ELEMENTWISE)
        with pytest.raises(ValueError):
            fn(desc, G, idx, off, None, W, rows.double(), 0.1, 1e-8, *extra)


def test_binding_checks_dense_arrays_before_any_call():
    desc = tbe.TBEDesc([10, 4], [8, 16], 2, device="cpu")
    idx = torch.zeros(3, dtype=torch.int64)
    off = torch.tensor([0, 1, 2, 2, 3], dtype=torch.int64)
    W = torch.zeros(desc.num_weights, dtype=torch.float16)
    with pytest.raises(ValueError):  # out of the wrong size
        tbe.tbe_forward(desc, W, idx, off, None, torch.empty(2, 23), None)
    with pytest.raises(ValueError):  # non-contiguous out
        tbe.tbe_forward(desc, W, idx, off, None, torch.empty(24, 2).t(), None)
    with pytest.raises(ValueError):  # one per-sample weight short
        tbe.tbe_forward(desc, W, idx, off, torch.ones(2), torch.empty(2, 24), None)
    with pytest.raises(ValueError):  # grad_out in fp64
        tbe.tbe_backward_rowwise_adagrad(desc, torch.zeros(2, 24, dtype=torch.float64), idx, off,
                                         None, W, torch.zeros(desc.total_E), 0.1, 1e-8, None)
