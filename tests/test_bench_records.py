"""The bench's DRAM-traffic records (host logic, no GPU).

A record of a kernel's DRAM bytes per work unit, scaled from a one-kernel
capture, counts only while the kernel's sources are those it was captured
on: a sha1 over whole files, or over a file's part before a marker line.
The bench then reports the bytes of a launch as units x bytes per unit, and
null otherwise.  Also the compulsory-byte model behind its problem roofline:
distinct valid rows per table, and how the forward, backward and step
counts relate."""
import hashlib
import os

import pytest

import bench
import table_embedding_bag_gb300 as tbe

CSRC = os.path.join(bench.ROOT, "table_embedding_bag_gb300", "csrc")


def test_sha_over_a_prefix_ends_at_the_marker():
    name, marker = bench.ROOFLINE_KERNELS["expand_count_kernel"]["sources"][0]
    text = open(os.path.join(CSRC, name), "rb").read()
    cut = text.find(marker.encode())
    assert cut > 0
    assert bench.source_sha1([(name, marker)]) == hashlib.sha1(text[:cut]).hexdigest()[:16]
    assert bench.source_sha1([name]) == hashlib.sha1(text).hexdigest()[:16]
    assert bench.source_sha1([name]) != bench.source_sha1([(name, marker)])


def test_sha_covers_every_file_in_order():
    a, b = "update.cu", "common.cuh"
    ta = open(os.path.join(CSRC, a), "rb").read()
    tb = open(os.path.join(CSRC, b), "rb").read()
    assert bench.source_sha1([a, b]) == hashlib.sha1(ta + tb).hexdigest()[:16]
    assert bench.source_sha1([a, b]) != bench.source_sha1([b, a])


def test_missing_marker_is_an_error():
    with pytest.raises(SystemExit):
        bench.source_sha1([("preprocess.cu", "// a line that is not in the file //")])


@pytest.mark.parametrize("name", list(bench.ROOFLINE_KERNELS))
def test_record_counts_only_for_its_sources(monkeypatch, name):
    k = bench.ROOFLINE_KERNELS[name]
    rec = dict(k["record"], source_sha1=bench.source_sha1(k["sources"]), bytes_per_unit=2.5)
    monkeypatch.setitem(k, "record", rec)
    assert bench.recorded_traffic(name, 1000) == 2500
    monkeypatch.setitem(k, "record", dict(rec, source_sha1="0" * 16))
    assert bench.recorded_traffic(name, 1000) is None
    monkeypatch.setitem(k, "record", None)
    assert bench.recorded_traffic(name, 1000) is None


def test_roofline_kernels_name_library_probes():
    assert bench.ROOFLINE_DOMINANT in bench.ROOFLINE_KERNELS
    for name, k in bench.ROOFLINE_KERNELS.items():
        assert isinstance(getattr(tbe, k["probe"]), int), name
        assert k["record"] is None or k["record"]["bytes_per_unit"] > 0


def test_rows_touched_counts_distinct_valid_rows():
    import workloads
    w = workloads.make("mixed", seed=2, B=128, T=4, E_scale=0.001)
    idx = w.indices.clone()
    idx[::7] = -1  # out-of-range rows are not rows
    w.indices = idx
    got = bench.rows_touched(w)
    off = w.offsets.numpy()
    for t in range(w.T):
        rows = idx.numpy()[off[t * w.B]:off[(t + 1) * w.B]]
        assert got[t] == len({int(r) for r in rows if 0 <= r < w.E[t]})


def test_compulsory_bytes_parts():
    import workloads
    w = workloads.make("weighted", seed=1, B=64, T=3, E_scale=0.001)
    rows = bench.rows_touched(w)
    c = bench.compulsory_bytes(w, rows, 4)
    dense = w.B * int(w.D.sum()) * 4
    rows_w = sum(int(r) * int(d) * 2 for r, d in zip(rows, w.D))
    # the step adds the output write to the backward; the backward adds the
    # rows' write and the momentum to the forward's reads
    assert c["step"] - c["backward"] == dense
    assert c["backward"] - c["forward"] == rows_w + 8 * int(sum(rows))
    ew = bench.compulsory_bytes(w, rows, 4, elementwise=True)
    assert ew["backward"] - c["backward"] == sum(int(r) * 8 * (int(d) - 1)
                                                 for r, d in zip(rows, w.D))
