"""TBE training-step benchmark: pooled forward + backward with row-wise Adagrad.

One step = tbe_preprocess (expand, radix sort, run-length encode, classify)
+ tbe_forward from the preprocessed workspace + tbe_backward_rowwise_adagrad
on the preprocessed runs (hot rows on the tensor cores, short-, medium- and
long-run update kernels), over one batch of the hot-row workload: T=8 tables
of E=1e7 rows, D=128, fp16 weights (20.5 GB) + fp32 row-wise momentum,
B=131072 bags per table, L=200 lookups per bag (209.7M lookups), Zipf(1.4)
rows over a per-table random permutation.  Several distinct batches are drawn
over the same tables (one table seed, per-batch draw seeds) and cycled, so
each step uses the hot set the backward learned on a different batch.
Inputs are drawn on the device once (seeded) and stay resident; every timed
step applies a real optimizer update.  Indices (1.7 GB per batch) and weights
(20.5 GB) are far larger than the 129 MB L2, so no flush is needed between
steps.

Besides the headline line it reports, per recipe of the workload set (tiny,
small, mixed, weighted, hot), forward / backward / step times in both
arrangements of the preprocessing, lookups/s and compulsory-byte roofline
fractions, and the long runs' fused and two-launch updates.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Rank 0 prints one JSON line.  With N > 1 (torchrun) every rank runs its own
independent batches (table seed = rank): weak scaling with no collective on
the data path; value = lookups of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import select
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TBE fwd+bwd lookups/sec (row-wise Adagrad) and achieved HBM GB/s vs GB300 peak"
WORKLOAD = ("hot-row: T=8 tables, E=1e7 rows, D=128, fp16 weights + fp32 row-wise momentum, "
            "B=131072 bags/table, L=200, Zipf(1.4) rows, unweighted, int64 indices, "
            "lr=0.01 eps=1e-8")
INDEX_BYTES = 8


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--cpu-bags", type=int, default=16384,
                   help="bags of table 0 in the CPU-oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-copy-streams", type=int, default=1,
                   help="copy streams sharing each step's host-to-device uploads in the e2e loop")
    p.add_argument("--batches", type=int, default=4,
                   help="distinct batches of the recipe cycled through the steps")
    p.add_argument("--configs", default="tiny,small,mixed,weighted,hot",
                   help="recipes measured for the per-config figures")
    p.add_argument("--config-steps", type=int, default=10)
    p.add_argument("--no-configs", action="store_true")
    p.add_argument("--pooling", choices=["sum", "mean"], default="sum",
                   help="pooling mode of the step (the recorded workload is sum)")
    p.add_argument("--weights", choices=["fp16", "bf16", "fp32"], default="fp16",
                   help="weight type (the recorded workload is fp16)")
    p.add_argument("--optimizer", choices=["rowwise", "elementwise"], default="rowwise",
                   help="Adagrad form (the recorded workload is row-wise)")
    # other recipes and smaller variants of one, for profiling captures only
    p.add_argument("--recipe", choices=["hot", "weighted", "mixed", "small", "tiny"],
                   default="hot")
    p.add_argument("--tables", type=int, default=None)
    p.add_argument("--rows", type=int, default=None)
    p.add_argument("--bags", type=int, default=None)
    return p.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "native" else "gloo"
        if args.impl == "native":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available() and args.impl == "native":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.first = ""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        # start timing only once sampling is live (its first line is out)
        ready, _, _ = select.select([self.proc.stdout], [], [], 5.0)
        if ready:
            self.first = self.proc.stdout.readline()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.first + out).strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# The roofline kernels: the largest steady-state shares of the step's
# kernels in the ncu launch list of this workload (distinct batches, hot set
# learned on the batch before; --cache-control none, so that the serialised
# per-launch times match the live probes): the expand of the preprocess
# (15.3 %), the cold-list forward (15.0 %) and the short-run update
# (14.6 %).  `roofline` reports the first, `roofline_kernels` the others.
# Each is timed live by the library's kernel probe.  A traffic record holds
# the DRAM bytes per work unit of one launch from a one-kernel ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum) of this recipe reduced to
# one table (each table is an independent draw and the kernels take the
# tables one after another), with the sha1 of the kernel's sources it was
# taken on: the bench scales it by the units of a full launch while the
# sources are unchanged, else reports null.
ROOFLINE_DOMINANT = "expand_count_kernel"
ROOFLINE_KERNELS = {
    "expand_count_kernel": {
        "what": "expand of tbe_preprocess: reads every index, writes the hot rows' byte "
                "histogram and the cold keys",
        "probe": "TBE_PROBE_EXPAND_COUNT",
        # the part of preprocess.cu up to the end of the kernel (its helpers
        # come before it), and common.cuh
        "sources": (("preprocess.cu", "// Compaction of the cold lookups"), "common.cuh"),
        "record": {"bytes_per_unit": 9.306, "unit": "lookup",
                   "source_sha1": "0f27c5bf3f9aaa36",
                   "capture": "hot-row recipe reduced to one table (E=1e7, D=128, B=131072), "
                              "two launches, dram__bytes_read.sum + dram__bytes_write.sum = "
                              "243.9 MB per launch over 26.21 M lookups"}},
    "forward_cold_piped_kernel": {
        "what": "cold-list forward of tbe_forward(TBE_F_PREPROCESSED): gathers the cold "
                "rows and adds them to the hot sums",
        "probe": "TBE_PROBE_FORWARD_COLD", "sources": ("forward.cu", "pool.cuh", "common.cuh"),
        "record": {"bytes_per_unit": 74.07, "unit": "cold lookup",
                   "source_sha1": "ad5f48928d886de1",
                   "capture": "hot-row recipe reduced to one table (E=1e7, D=128, B=131072), "
                              "two launches, dram__bytes_read.sum + dram__bytes_write.sum = "
                              "167.6 MB per launch over 2.263 M cold lookups"}},
    "short_runs_kernel": {
        "what": "short-run update of tbe_backward_rowwise_adagrad (runs of fewer than 16 "
                "pairs)",
        "probe": "TBE_PROBE_SHORT_RUNS", "sources": ("update.cu", "common.cuh"),
        "record": {"bytes_per_unit": 495.72, "unit": "short-run pair",
                   "source_sha1": "c4fe9027c6c98b56",
                   "capture": "hot-row recipe reduced to one table (E=1e7, D=128, B=131072), "
                              "two launches, dram__bytes_read.sum + dram__bytes_write.sum = "
                              "219.3 MB per launch over 442 434 short-run pairs"}},
}


def source_sha1(files):
    """First 16 hex digits of the sha1 over a kernel's sources: whole files,
    or (file, marker) for the part of a file before the marker line."""
    import hashlib
    h = hashlib.sha1()
    for f in files:
        name, marker = (f, None) if isinstance(f, str) else f
        text = open(os.path.join(ROOT, "table_embedding_bag_gb300", "csrc", name), "rb").read()
        if marker is not None:
            cut = text.find(marker.encode())
            if cut < 0:
                raise SystemExit(f"bench: marker {marker!r} not found in {name}")
            text = text[:cut]
        h.update(text)
    return h.hexdigest()[:16]


def recorded_traffic(name, units):
    """DRAM bytes of one launch of kernel `name` over `units` work units,
    scaled from its recorded capture; None without a record of the current
    sources."""
    k = ROOFLINE_KERNELS[name]
    rec = k["record"]
    if rec is None or rec["source_sha1"] != source_sha1(k["sources"]):
        return None
    return int(rec["bytes_per_unit"] * units)


def workload_name(args, base=WORKLOAD):
    """The workload string with the step's weight type, Adagrad form and
    pooling."""
    ew = args.optimizer == "elementwise"
    return (base.replace("fp16 weights", f"{args.weights} weights").replace(
        "row-wise momentum",
        "per-element momentum (element-wise Adagrad)" if ew else "row-wise momentum") +
        (", mean pooling" if args.pooling == "mean" else ""))


def momentum_bytes(D, elementwise):
    """Momentum bytes a row's update reads and writes: one fp32 per row, or
    one per element with element-wise Adagrad."""
    return 8 * D if elementwise else 8


def short_run_bytes(D, pairs, runs, all_runs, elementwise=False, wb=2):
    """Algorithmic bytes of one short_runs_kernel launch, counted per use: per
    short-run pair its bag (4), pair start (8) and gradient row (4 D); per
    short run the weights row read and written (2 x wb D, wb bytes per
    weight) and the momentum (8, or 8 D element-wise); per run of the batch
    its run data (8: the kernel walks every run to pick the short ones)."""
    return (pairs * (4 + 8 + 4 * D) + runs * (2 * wb * D + momentum_bytes(D, elementwise))
            + all_runs * 8)


def expand_bytes(w, units, per_use=True):
    """Bytes of one expand_count_kernel launch: every index (and per-sample
    weight) read once and each bag's offset; the hot rows' histogram row of
    every bag of a table with hot rows written (a byte per slot, fp32 with
    per-sample weights); each cold key (and weight) and each bag's cold count
    written.  Per use it adds each CTA's read of its table's hot set (kHot
    keys and places), which L2 serves after the first."""
    nb = w.T * w.B
    psw = w.psw is not None
    b = (w.n * w.indices.element_size() + (nb + 1) * w.offsets.element_size()
         + (4 * w.n if psw else 0))
    b += units["hot_tables"] * w.B * 256 * (4 if psw else 1)
    b += units["cold_lookups"] * (8 if psw else 4) + nb * 4
    if per_use:
        b += w.T * ((w.B + 127) // 128) * 256 * 8
    return int(b)


def cold_forward_bytes(w, units, D):
    """Per-use bytes of one forward_cold_piped_kernel launch: per cold lookup
    its key (4, + 4 weight) and its row (D weights); per bag its list offset
    (4) and its fp32 output row, read and written where the bag's table has
    hot rows (the hot forward pooled them first), else written."""
    nb = w.T * w.B
    wb = w.weights.element_size()
    per = 4 + (4 if w.psw is not None else 0) + wb * D
    return int(units["cold_lookups"] * per + (nb + 1) * 4
               + units["hot_tables"] * w.B * 8 * D + (w.T - units["hot_tables"]) * w.B * 4 * D)


def compulsory_bytes(w, rows_touched, index_bytes, elementwise=False):
    """Compulsory bytes of the forward, the backward and the whole step of
    batch w: every index, offset and per-sample weight read once, every
    distinct row once (rows_touched[t] rows of table t), the pooled output
    written once and its gradient read once, each touched row's weights and
    momentum read and written once."""
    nb = w.T * w.B
    idx = w.n * index_bytes + (nb + 1) * index_bytes + (4 * w.n if w.psw is not None else 0)
    dense = w.B * int(w.D.sum()) * 4
    rows_w = sum(int(r) * int(d) * w.weights.element_size() for r, d in zip(rows_touched, w.D))
    rows_m = sum(int(r) * momentum_bytes(int(d), elementwise) for r, d in zip(rows_touched, w.D))
    return {"forward": idx + rows_w + dense,
            "backward": idx + dense + 2 * rows_w + rows_m,
            "step": idx + 2 * dense + 2 * rows_w + rows_m}


def rows_touched(w):
    """Distinct valid rows each table's lookups touch (on the device)."""
    L = (w.offsets[1:] - w.offsets[:-1]).long()
    t_of = torch.repeat_interleave(torch.arange(w.T * w.B, device=L.device) // w.B, L)
    E = torch.as_tensor(w.E, device=L.device)
    r = w.indices.long()
    ok = (r >= 0) & (r < E[t_of])
    hb = torch.as_tensor(np.concatenate([[0], np.cumsum(w.E)]), device=L.device)
    keys = torch.unique(hb[t_of[ok]] + r[ok])
    return torch.bincount(torch.searchsorted(hb[1:], keys, right=True), minlength=w.T).cpu().numpy()


def draw_batches(name, dev, rank, K, **kw):
    """K distinct batches over one set of tables (table seed = rank): the
    first drawn with its weights, the others sharing them."""
    import workloads
    w0 = workloads.make(name, device=dev, seed=1000 * rank, table_seed=rank, **kw)
    return [w0] + [workloads.batch(w0, 1000 * rank + k) for k in range(1, K)]


class Stepper:
    """One problem's state (descriptor, workspace, weights, momentum, output)
    and its training step through the public API."""

    def __init__(self, tbe, batches, dev, wdt=torch.float16, mean=False, elementwise=False,
                 momentum=None):
        w = batches[0]
        self.tbe = tbe
        self.weighted = w.psw is not None
        self.desc = tbe.TBEDesc(w.E, w.D, w.B, w.indices.dtype, dev, wdt)
        self.n_max = max(b.n for b in batches)
        self.ws = tbe.Workspace(self.desc, max(self.n_max, 1), self.weighted, dev, mean=mean)
        self.weights = w.weights
        self.momentum = momentum if momentum is not None else (
            torch.zeros(self.desc.num_weights, dtype=torch.float32, device=dev) if elementwise
            else w.momentum)
        self.out = torch.empty(w.B, self.desc.total_D, dtype=torch.float32, device=dev)
        self.pre_flags = tbe.TBE_F_PREPROCESSED | (tbe.TBE_F_MEAN if mean else 0)
        self.upd_flags = self.pre_flags | (tbe.TBE_F_ELEMENTWISE if elementwise else 0)
        self.mean = mean
        self.elementwise = elementwise

    def step(self, w, ev=None, arrangement="pre_in_fwd", two_launch=False):
        """One training step on batch w.  pre_in_fwd (the timed step): one
        preprocess of the batch serves the forward and the backward;
        pre_in_bwd: the plain forward from the indices, and the backward
        with its own preprocess.  ev: four events recorded around the
        phases (pre_in_bwd: its first two coincide)."""
        tbe = self.tbe
        s = torch.cuda.current_stream()
        extra = tbe.TBE_F_LONG_TWO_LAUNCH if two_launch else 0
        rec = (lambda i: ev[i].record(s)) if ev is not None else (lambda i: None)
        rec(0)
        if arrangement == "pre_in_fwd":
            tbe.tbe_preprocess(self.desc, w.indices, w.offsets, w.psw, self.ws)
            rec(1)
            tbe.tbe_forward(self.desc, self.weights, w.indices, w.offsets, w.psw, self.out,
                            self.ws, self.pre_flags)
            rec(2)
            tbe.tbe_backward_rowwise_adagrad(self.desc, w.grad_out, w.indices, w.offsets, w.psw,
                                             self.weights, self.momentum, w.lr, w.eps, self.ws,
                                             self.upd_flags | extra)
        else:
            rec(1)
            plain = (tbe.TBE_F_MEAN if self.mean else 0)
            tbe.tbe_forward(self.desc, self.weights, w.indices, w.offsets, w.psw, self.out,
                            self.ws, plain)
            rec(2)
            tbe.tbe_backward_rowwise_adagrad(
                self.desc, w.grad_out, w.indices, w.offsets, w.psw, self.weights, self.momentum,
                w.lr, w.eps, self.ws, plain | (tbe.TBE_F_ELEMENTWISE if self.elementwise else 0)
                | extra)
        rec(3)

    def counters(self):
        """The workspace's device counters after the last preprocess (syncs)."""
        torch.cuda.synchronize()
        v = self.tbe.tbe_workspace_view(self.desc, self.n_max, self.ws)
        o = v["counts"] - self.ws.buf.data_ptr()
        return self.ws.buf[o:o + 36].view(torch.int32).cpu().numpy().view(np.uint32), v

    def ws_u32(self, ptr, count):
        o = ptr - self.ws.buf.data_ptr()
        return self.ws.buf[o:o + 4 * count].view(torch.int32)

    def clear_hot_set(self):
        """Empty the hot set the next preprocess takes (as in a fresh workspace)."""
        torch.cuda.synchronize()
        v = self.tbe.tbe_workspace_view(self.desc, self.n_max, self.ws)
        self.ws_u32(v["hot_n"], self.desc.T).zero_()
        torch.cuda.synchronize()


def run_units(st, w):
    """Work units of the last backward on batch w (counters of its
    preprocess): cold lookups, runs by class, short-run pairs, and the
    distinct (table, bag) gradient rows the short runs gather."""
    c, v = st.counters()
    R, n_long, n_chunks, n_cold = int(c[0]), int(c[2]), int(c[3]), int(c[7])
    rp = st.ws_u32(v["run_pairs"], R + 1).long()
    sl = rp[1:] - rp[:-1]
    short = sl < int(v["medium_threshold"])
    lng = sl >= int(v["long_threshold"])
    P = int(c[6])
    pair_run = torch.repeat_interleave(torch.arange(R, device=rp.device), sl)
    pb = st.ws_u32(v["pair_bags"], P).long()
    uk = st.ws_u32(v["unique_keys"], R).long() & 0xffffffff
    hb = torch.as_tensor(np.concatenate([[0], np.cumsum(w.E)]), device=rp.device)
    t_run = torch.searchsorted(hb[1:], uk, right=True)
    sp = short[pair_run]
    short_bag_rows = int(torch.unique(t_run[pair_run[sp]] * w.B + pb[sp]).numel())
    hot_n = st.ws_u32(v["hot_n"], w.T)
    hn = int(hot_n.sum().item())
    return {"R": R, "long_runs": n_long, "long_chunks": n_chunks, "cold_lookups": n_cold,
            "hot_tables": int((hot_n > 0).sum().item()),
            "short_runs": int(short.sum().item()), "short_pairs": int(sl[short].sum().item()),
            "long_pairs": int(sl[lng].sum().item()), "short_bag_rows": short_bag_rows,
            "hot_rows_next": hn, "hit_rate": 1.0 - n_cold / max(w.n, 1)}


def l2_flush(buf):
    """Overwrite a buffer larger than L2 (outside the timed events)."""
    if buf is not None:
        buf.add_(1)


def time_phases(st, batches, steps, warmup, arrangement="pre_in_fwd", two_launch=False,
                flush=None, first=0):
    """Median phase times (ms) over `steps` timed steps cycling the batches
    (warm-up steps first; every step's hot set comes from the step before)."""
    K = len(batches)
    for k in range(warmup):
        st.step(batches[(first + k) % K], arrangement=arrangement, two_launch=two_launch)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for k in range(steps):
        l2_flush(flush)
        st.step(batches[(first + warmup + k) % K], evs[k], arrangement, two_launch)
    torch.cuda.synchronize()
    ph = lambda a, b: statistics.median(e[a].elapsed_time(e[b]) for e in evs)
    return {"pre_ms": ph(0, 1), "fwd_ms": ph(0, 2), "bwd_ms": ph(2, 3), "step_ms": ph(0, 3),
            "next": first + warmup + steps}


CONFIG_KW = {"tiny": {}, "small": {}, "mixed": {}, "weighted": {}, "hot": {}}


def time_graph_steps(st, batches, steps, warmup, flush=None):
    """Median step time (ms) with each batch's whole step (preprocess,
    forward, backward) captured once into a CUDA graph and the graphs
    replayed in turn: the same kernels without the host's per-launch cost."""
    K = len(batches)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graphs = []
    for b in batches:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                st.step(b)
        graphs.append(g)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    for k in range(warmup):
        graphs[k % K].replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for k in range(steps):
        l2_flush(flush)
        evs[k][0].record(s)
        graphs[k % K].replay()
        evs[k][1].record(s)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def measure_configs(tbe, dev, rank, args, hbm, main=None):
    """Per recipe at its stated size: forward, backward and step ms in both
    arrangements of the preprocessing (in the forward: one preprocess serves
    both passes; in the backward: the plain forward from the indices and a
    backward that sorts for itself), lookups/s, and the compulsory bytes of
    each phase as a fraction of the HBM peak; for the hot and weighted
    recipes also the long runs' fused and two-launch updates.  L2 is flushed
    before every timed step.  main: the hot recipe's batches and stepper of
    the headline run, reused."""
    res = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # 2x L2
    for name in args.configs.split(","):
        if name == "hot" and main is not None:
            batches, st = main
        else:
            batches = draw_batches(name, dev, rank, 2, **CONFIG_KW[name])
            st = Stepper(tbe, batches, dev)
        w = batches[0]
        ib = w.indices.element_size()
        steps, warm = args.config_steps, 3
        r = {"n_lookups": w.n, "T": w.T, "B": w.B}
        touched = rows_touched(w)
        cb = compulsory_bytes(w, touched, ib)
        first = 0
        for arr in ("pre_in_fwd", "pre_in_bwd"):
            ph = time_phases(st, batches, steps, warm, arr, flush=flush, first=first)
            first = ph["next"]
            r[arr] = {"fwd_ms": ph["fwd_ms"], "bwd_ms": ph["bwd_ms"], "sum_ms": ph["step_ms"],
                      "lookups_per_s": w.n / (ph["step_ms"] / 1e3),
                      "roofline_frac": {k: cb[k] / (t / 1e3) / 1e9 / hbm for k, t in
                                        (("forward", ph["fwd_ms"]), ("backward", ph["bwd_ms"]),
                                         ("step", ph["step_ms"]))}}
        if name in ("tiny", "small", "mixed"):
            # launch-bound recipes: the same step replayed as a CUDA graph
            g_ms = time_graph_steps(st, batches, steps, warm, flush=flush)
            r["graph"] = {"sum_ms": g_ms, "lookups_per_s": w.n / (g_ms / 1e3),
                          "note": "each batch's step captured once into a CUDA graph "
                                  "and replayed"}
        if name in ("hot", "weighted"):
            ph2 = time_phases(st, batches, steps, warm, "pre_in_fwd", two_launch=True,
                              flush=flush, first=first)
            r["long_runs_update"] = {"fused_bwd_ms": r["pre_in_fwd"]["bwd_ms"],
                                     "two_launch_bwd_ms": ph2["bwd_ms"],
                                     "two_launch_sum_ms": ph2["step_ms"]}
        r["compulsory_bytes"] = cb
        res[name] = r
        if not (name == "hot" and main is not None):
            del st, batches, w
            torch.cuda.empty_cache()
    r0 = {"note": "median of timed steps over 2 distinct batches per recipe (the hot recipe: "
                  "the headline batches); fractions are compulsory bytes over time against "
                  "the measured HBM peak; L2 flushed before each timed step"}
    res.update(r0)
    return res


def run_native(args, world, rank, local):
    import table_embedding_bag_gb300 as tbe

    dev = torch.device("cuda", torch.cuda.current_device())
    import workloads
    E_scale = None if args.rows is None else args.rows / workloads.SPECS["hot"].E
    if args.recipe != "hot" and args.rows is not None:
        raise SystemExit("--rows applies to the hot-row recipe only")
    wdt = {"bf16": torch.bfloat16, "fp32": torch.float32}.get(args.weights, torch.float16)
    mean = args.pooling == "mean"
    ew = args.optimizer == "elementwise"
    K = max(1, args.batches)
    batches = draw_batches(args.recipe, dev, rank, K, T=args.tables, B=args.bags,
                           E_scale=E_scale, weights_dtype=wdt)
    w = batches[0]
    st = Stepper(tbe, batches, dev, wdt, mean=mean, elementwise=ew)
    stream = torch.cuda.current_stream()

    for k in range(args.warmup):
        st.step(batches[k % K])
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = Clocks(local)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    tbe.tbe_probe_set(tbe.TBE_PROBE_SHORT_RUNS)
    launches0 = tbe.tbe_kernel_launches()
    t0.record(stream)
    for k in range(args.steps):
        st.step(batches[(args.warmup + k) % K], evs[k])
    t1.record(stream)
    launches = tbe.tbe_kernel_launches() - launches0
    probe_launches, probe_ms = tbe.tbe_probe_read()
    tbe.tbe_probe_set(tbe.TBE_PROBE_OFF)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    status = tbe.tbe_read_status(st.ws)
    if status & tbe.TBE_ERR_TIMEOUT:
        raise SystemExit("bench: a kernel's bounded wait timed out during the timed steps "
                         f"(status {status:#x}); the measurement is invalid")
    ms_local = t0.elapsed_time(t1)
    ms = max_over_ranks(ms_local, world, dev)
    pre = [e[0].elapsed_time(e[1]) for e in evs]
    fwd = [e[1].elapsed_time(e[2]) for e in evs]
    upd = [e[2].elapsed_time(e[3]) for e in evs]
    lookups = sum(batches[(args.warmup + k) % K].n for k in range(args.steps))

    # work units per batch, continuing the cycle (each hot set from the batch before)
    nxt = args.warmup + args.steps
    units = []
    for j in range(K):
        b = batches[(nxt + j) % K]
        st.step(b)
        units.append(run_units(st, b))
    nxt += K
    avg = {k: float(np.mean([u[k] for u in units])) for k in units[0]}
    # the other roofline kernels timed live by the probe (2 K steps each,
    # continuing the cycle)
    probes = {"short_runs_kernel": (probe_launches, probe_ms)}
    for name in ("expand_count_kernel", "forward_cold_piped_kernel"):
        tbe.tbe_probe_set(getattr(tbe, ROOFLINE_KERNELS[name]["probe"]))
        for j in range(2 * K):
            st.step(batches[(nxt + j) % K])
        nxt += 2 * K
        probes[name] = tbe.tbe_probe_read()
        tbe.tbe_probe_set(tbe.TBE_PROBE_OFF)
    # first step with an empty hot set (a fresh workspace's first batch)
    st.clear_hot_set()
    ce = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    b = batches[nxt % K]
    st.step(b, ce)
    torch.cuda.synchronize()
    cold = {"step_ms": ce[0].elapsed_time(ce[3]), "fwd_ms": ce[0].elapsed_time(ce[2]),
            "bwd_ms": ce[2].elapsed_time(ce[3])}
    nxt += 1
    result = {
        "ms": ms, "ms_local": ms_local, "fwd_ms": statistics.median(fwd),
        "pre_ms": statistics.median(pre), "upd_ms": statistics.median(upd),
        "lookups": lookups, "units": avg, "units_per_batch": units, "cold_start": cold,
        "clocks": clk, "probe_launches": probe_launches, "probe_ms": probe_ms, "probes": probes,
        "launches": launches, "w": w, "batches": batches, "stepper": st, "next": nxt,
    }

    if not args.no_e2e:
        # End to end through the public API: per step, this step's inputs go
        # host -> device from pinned memory and the pooled output comes back.
        # Two distinct batches alternate on the host.  Two device input slots:
        # step k+1's uploads (copy stream) overlap step k's compute, and step
        # k's output download (a third stream) overlaps its backward; every
        # copy stays inside the timed region.
        hb = [(b.indices.cpu().pin_memory(), b.offsets.cpu().pin_memory(),
               b.grad_out.cpu().pin_memory()) for b in batches[:2]]
        out = st.out
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        slots = [(torch.empty_like(w.indices), torch.empty_like(w.offsets),
                  torch.empty_like(w.grad_out)) for _ in range(2)]
        # the uploads are split into contiguous pieces on several copy
        # streams, so that several copy engines share the host link
        nup = max(1, args.e2e_copy_streams)
        ups = [torch.cuda.Stream() for _ in range(nup)]
        down = torch.cuda.Stream()
        copied = [[torch.cuda.Event() for _ in range(nup)] for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        fwd_done, out_read = torch.cuda.Event(), torch.cuda.Event()

        def pieces(t):
            f = t.view(-1)
            step = (f.numel() + nup - 1) // nup
            return [f[i * step:(i + 1) * step] for i in range(nup)]

        def e2e_step(k):
            d_idx, d_off, d_grad = slots[k % 2]
            h_idx, h_off, h_grad = hb[k % len(hb)]
            parts = [list(zip(pieces(d), pieces(h)))
                     for d, h in ((d_idx, h_idx), (d_off, h_off), (d_grad, h_grad))]
            for j, up in enumerate(ups):
                with torch.cuda.stream(up):
                    if k >= 2:
                        up.wait_event(consumed[k % 2])
                    for pr in parts:
                        if pr[j][0].numel():
                            pr[j][0].copy_(pr[j][1], non_blocking=True)
                    copied[k % 2][j].record(up)
            for ev in copied[k % 2]:
                stream.wait_event(ev)
            if k >= 1:
                stream.wait_event(out_read)  # the previous output was read back
            tbe.tbe_preprocess(st.desc, d_idx, d_off, None, st.ws)
            tbe.tbe_forward(st.desc, st.weights, d_idx, d_off, None, out, st.ws, st.pre_flags)
            fwd_done.record(stream)
            with torch.cuda.stream(down):
                down.wait_event(fwd_done)
                h_out.copy_(out, non_blocking=True)
                out_read.record(down)
            tbe.tbe_backward_rowwise_adagrad(st.desc, d_grad, d_idx, d_off, None, st.weights,
                                             st.momentum, w.lr, w.eps, st.ws, st.upd_flags)
            consumed[k % 2].record(stream)

        for k in range(max(1, args.warmup)):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier(world)
        a = torch.cuda.Event(enable_timing=True)
        bev = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for up in ups:
            up.wait_event(a)
        down.wait_event(a)
        for k in range(args.steps):
            e2e_step(k + 2 * args.warmup)  # the slot pattern continues past the warm-up
        stream.wait_event(out_read)
        bev.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(a.elapsed_time(bev), world, dev)
        result["e2e_ms"] = e2e_ms
        result["e2e_lookups"] = sum(batches[(k + 2 * args.warmup) % len(hb)].n
                                    for k in range(args.steps))
        hidx, hoff, hgrad = hb[0]
        result["h2d"] = (hidx.numel() * hidx.element_size() + hoff.numel() * hoff.element_size()
                         + hgrad.numel() * 4)
        result["d2h"] = h_out.numel() * 4
        result["e2e_copy_streams"] = nup
        # the host link as this process sees it, for context: one step's
        # uploads (all on one stream) and its download, each alone, best of
        # three; the e2e step cannot be shorter than the slower direction
        d_idx, d_off, d_grad = slots[0]
        h_idx, h_off, h_grad = hb[0]
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        up_ms, down_ms = [], []
        for _ in range(3):
            ev[0].record(stream)
            for d, h in ((d_idx, h_idx), (d_off, h_off), (d_grad, h_grad)):
                d.copy_(h, non_blocking=True)
            ev[1].record(stream)
            torch.cuda.synchronize()
            up_ms.append(ev[0].elapsed_time(ev[1]))
            ev[0].record(stream)
            h_out.copy_(out, non_blocking=True)
            ev[1].record(stream)
            torch.cuda.synchronize()
            down_ms.append(ev[0].elapsed_time(ev[1]))
        result["link"] = {"h2d_GBps": result["h2d"] / min(up_ms) / 1e6,
                          "d2h_GBps": result["d2h"] / min(down_ms) / 1e6,
                          "h2d_ms": min(up_ms), "d2h_ms": min(down_ms)}
        del hb, slots
    return result


def cpu_sample(w_dev, bags, first=0):
    """Table 0, its bags [first, first + bags), as a standalone host problem
    holding only the rows those bags touch (renumbered)."""
    import workloads
    off = w_dev.offsets[first:first + bags + 1].cpu().numpy().astype(np.int64)
    idx_dev = w_dev.indices[int(off[0]):int(off[-1])]
    off = off - off[0]
    uniq, inv = torch.unique(idx_dev, return_inverse=True)
    D0 = int(w_dev.D[0])
    rows = w_dev.weights[:int(w_dev.E[0]) * D0].view(-1, D0)[uniq].cpu().reshape(-1)
    if rows.dtype != torch.bfloat16:
        rows = rows.numpy()
    G0 = w_dev.grad_out[first:first + bags, :D0].cpu().numpy()
    E0 = int(uniq.numel())
    return workloads.from_arrays([E0], [D0], bags, inv.cpu().numpy(), off, rows, G0,
                                 momentum=np.zeros(E0, np.float32), lr=w_dev.lr, eps=w_dev.eps)


def time_oracle(s, mean=False, elementwise=False):
    """Seconds the oracle takes for one forward and backward of sample s, in
    the step's pooling, weight type and Adagrad form."""
    import oracle
    oracle.build()
    tab = oracle.Tables(s.E, s.D)
    idx, off = s.indices.numpy(), s.offsets.numpy()
    bf16 = s.weights.dtype == torch.bfloat16
    fp32 = s.weights.dtype == torch.float32
    W = s.weights.view(torch.int16).numpy().view(np.uint16) if bf16 else s.weights.numpy()
    G = s.grad_out.numpy()
    m = (np.zeros(int(tab.w_offsets[-1]), np.float32) if elementwise
         else s.momentum.numpy())
    t = time.perf_counter()
    oracle.forward(tab, s.B, W, idx, off, mean=mean, bf16=bf16, fp32=fp32)
    oracle.backward_rowwise_adagrad(tab, s.B, idx, off, G, W, m, s.lr, s.eps, mean=mean,
                                    bf16=bf16, elementwise=elementwise, fp32=fp32)
    return time.perf_counter() - t


def _oracle_worker(arrays):
    """One host core's share of the CPU baseline: the oracle on one sample
    (arrays of a workloads.from_arrays problem), timed in this process."""
    import workloads
    E, D, B, idx, off, W, G, lr, eps, mean, ew = arrays
    s = workloads.from_arrays(E, D, B, idx, off, W, G, momentum=np.zeros(int(E[0]), np.float32),
                              lr=lr, eps=eps)
    return time_oracle(s, mean, ew), s.n


def cpu_baseline_parallel(w, bags, cores, mean=False, elementwise=False):
    """The oracle, as it stands, on `cores` disjoint samples of table 0 of
    batch w (bags [k bags, (k + 1) bags) for core k), one process per host
    core started by spawn; lookups of all samples over the wall time of the
    slowest.  Returns (lookups/s, lookups, seconds)."""
    import multiprocessing as mp
    jobs = []
    for k in range(cores):
        s = cpu_sample(w, bags, first=k * bags)
        W = s.weights.numpy() if s.weights.dtype != torch.bfloat16 else s.weights
        jobs.append((s.E, s.D, s.B, s.indices.numpy(), s.offsets.numpy(), W, s.grad_out.numpy(),
                     s.lr, s.eps, mean, elementwise))
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_worker, jobs)
    secs = max(t for t, _ in res)
    n = sum(k for _, k in res)
    return n / secs, n, secs


def _openmp_worker(job):
    """The oracle's OpenMP form on one sample with `threads` threads, timed
    in this (spawned) process: (seconds, lookups, threads) or (None, reason,
    0) if it could not be built or run here."""
    threads, E, D, B, idx, off, W, G, lr, eps, mean, ew, bf16, fp32 = job
    try:
        import oracle
        import oracle.openmp as omp
        omp.build()
        omp.set_threads(threads)
        tab = oracle.Tables(E, D)
        m = np.zeros(int(tab.w_offsets[-1]) if ew else int(tab.hash_base[-1]), np.float32)
        t = time.perf_counter()
        omp.forward(tab, B, W, idx, off, mean=mean, bf16=bf16, fp32=fp32)
        omp.backward_rowwise_adagrad(tab, B, idx, off, G, W, m, lr, eps, mean=mean, bf16=bf16,
                                     elementwise=ew, fp32=fp32)
        return time.perf_counter() - t, len(idx), omp.threads()
    except Exception as e:  # a host without OpenMP: reported, not fatal
        return None, f"{type(e).__name__}: {e}"[:200], 0


def cpu_baseline_openmp(w, bags, cores, mean=False, elementwise=False):
    """The oracle's OpenMP form (forward parallel over bags, backward over the
    rows of the run map after a parallel sort) on bags [0, bags) of table 0
    of batch w, with one thread per host core, in a spawned process."""
    try:
        return _cpu_baseline_openmp(w, bags, cores, mean, elementwise)
    except Exception as e:  # reported, not fatal: the line is printed either way
        return {"value": None, "reason": f"{type(e).__name__}: {e}"[:200]}


def _cpu_baseline_openmp(w, bags, cores, mean, elementwise):
    import multiprocessing as mp
    s = cpu_sample(w, bags)
    bf16 = s.weights.dtype == torch.bfloat16
    fp32 = s.weights.dtype == torch.float32
    W = s.weights.view(torch.int16).numpy().view(np.uint16) if bf16 else s.weights.numpy()
    job = (cores, s.E, s.D, s.B, s.indices.numpy(), s.offsets.numpy(), W, s.grad_out.numpy(),
           s.lr, s.eps, mean, elementwise, bf16, fp32)
    with mp.get_context("spawn").Pool(1) as pool:  # left with terminate() on a time-out
        secs, n, threads = pool.apply_async(_openmp_worker, (job,)).get(timeout=120)
    if secs is None:
        return {"value": None, "reason": n}
    return {"value": n / secs, "unit": "lookups/s", "threads": threads,
            "kind": "oracle, OpenMP form (bit-identical results)",
            "sample": f"table 0 of the first batch, bags [0, {bags}) ({n} lookups), forward "
                      f"+ backward, {secs:.1f} s wall"}


def _reference_worker(job):
    """One host core's share of a reference-arm step: draw its own sample of
    the recipe and time the oracle on it (the draw is not timed)."""
    seed, bags, wname, mean, ew = job
    wdt = {"bf16": torch.bfloat16, "fp32": torch.float32}.get(wname, torch.float16)
    s = reference_sample(bags, seed=seed, weights_dtype=wdt)
    return time_oracle(s, mean, ew), s.n


def reference_sample(bags, seed=0, weights_dtype=torch.float16):
    """The same recipe's table 0, drawn on the host: bags x 200 lookups, with
    only the touched rows materialised."""
    import workloads
    return workloads.make("hot", device="cpu", seed=seed, B=bags, T=1, compact=True,
                          weights_dtype=weights_dtype)


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        if rank != 0:
            return
        import multiprocessing as mp
        bags = 2048
        cores = max(1, os.cpu_count() or 1)
        mean, ew = args.pooling == "mean", args.optimizer == "elementwise"
        times, lookups = [], 0
        with mp.get_context("spawn").Pool(cores) as pool:
            for k in range(args.warmup + args.steps):
                res = pool.map(_reference_worker, [(k * cores + i, bags, args.weights, mean, ew)
                                                   for i in range(cores)])
                if k >= args.warmup:
                    times.append(max(t for t, _ in res))  # the step ends with its slowest core
                    lookups += sum(n for _, n in res)
        tot = sum(times)
        value = lookups / tot
        line = {
            "impl": "reference", "metric": METRIC, "value": value, "unit": "lookups/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(args), "sample": f"per step, {cores} samples "
                                                     f"of table 0, {bags} bags x 200 lookups "
                                                     "each (same recipe, host-drawn, touched "
                                                     "rows only), one per host core"},
            "cpu_baseline": {"value": value, "unit": "lookups/s", "cores": cores, "kind": "oracle",
                             "sample": f"per step {cores} samples of table 0 of the hot-row "
                                       f"recipe, {bags} bags x 200 lookups each, forward + "
                                       "backward, one oracle process per core"},
            "e2e": {"value": value, "unit": "lookups/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return

    r = run_native(args, world, rank, local)
    w = r["w"]
    total_lookups = r["lookups"] * world
    value = total_lookups / (r["ms"] / 1e3)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    # row width of the byte models: the recipe's D, or (mixed widths) the
    # lookup-weighted mean width
    L_t = (w.offsets[1:].long() - w.offsets[:-1].long()).view(w.T, w.B).sum(1).cpu().numpy()
    D = int(round(float((L_t * w.D).sum() / max(L_t.sum(), 1))))
    ew = args.optimizer == "elementwise"
    u = r["units"]
    wb = w.weights.element_size()
    reduced = (args.tables, args.rows, args.bags) != (None,) * 3 or args.recipe != "hot"

    def kernel_entry(name, per_use, minimum, units, unit_name, model):
        launches, total_ms = r["probes"][name]
        if launches == 0:  # not part of this step (fp32 weights take no cold-list forward)
            return {"kernel": name, "what": ROOFLINE_KERNELS[name]["what"], "bound": "hbm",
                    "achieved": None, "peak": hbm, "unit": "GB/s", "frac": None,
                    "traffic": None, "launches_timed": 0, "note": "not launched by this step"}
        launch_ms = total_ms / max(launches, 1)
        ach = per_use / (launch_ms / 1e3) / 1e9
        e = {"kernel": name, "what": ROOFLINE_KERNELS[name]["what"], "bound": "hbm",
             "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
             "traffic": None if reduced else recorded_traffic(name, units),
             "peak_source": peak_src, "bytes_model": model, "bytes_per_launch": per_use,
             "launch_ms": launch_ms, "launches_timed": launches, "units": {unit_name: units}}
        if minimum is not None:
            e["compulsory_bytes_per_launch"] = minimum
            e["compulsory_frac"] = minimum / (launch_ms / 1e3) / 1e9 / hbm
        return e

    # compulsory bytes of the short runs: each short run's row and momentum
    # read and written once, its pair data once, each gradient row it
    # gathers once
    k_min = (u["short_runs"] * (2 * wb * D + momentum_bytes(D, ew)) + u["R"] * 8
             + u["short_pairs"] * 12 + u["short_bag_rows"] * 4 * D)
    kernels = {
        "expand_count_kernel": kernel_entry(
            "expand_count_kernel", expand_bytes(w, u), expand_bytes(w, u, per_use=False), w.n,
            "lookups", "per use: every index and offset, the histogram row of every bag of a "
                       "table with hot rows, the cold keys and counts, each CTA's hot-set "
                       "read"),
        "forward_cold_piped_kernel": kernel_entry(
            "forward_cold_piped_kernel", cold_forward_bytes(w, u, D), None, u["cold_lookups"],
            "cold_lookups", "per use: key and row per cold lookup, list offset and output "
                            "row read and written per bag"),
        "short_runs_kernel": kernel_entry(
            "short_runs_kernel", short_run_bytes(D, u["short_pairs"], u["short_runs"], u["R"],
                                                 ew, wb),
            k_min, u["short_pairs"], "short_pairs",
            "per use: bag + pair start + gradient row per short-run pair, weights row r/w + "
            "momentum per short run, run data per run"),
    }
    kernels["short_runs_kernel"]["units"].update(
        {"short_runs": u["short_runs"], "runs": u["R"], "short_bag_rows": u["short_bag_rows"]})
    touched = rows_touched(w)
    cb = compulsory_bytes(w, touched, w.indices.element_size(), ew)
    t_fwd = r["pre_ms"] + r["fwd_ms"]
    t_step = r["ms_local"] / args.steps
    t_bwd = r["upd_ms"]
    line = {
        "metric": METRIC, "value": value, "unit": "lookups/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_name(
                       args, WORKLOAD if not reduced
                       else f"{args.recipe} recipe T={w.T} B={w.B} n={w.n}"
                            + (" (reduced)" if args.recipe == "hot" else "")
                            + " (profiling case)"),
                   "n_lookups": w.n, "global_batch": w.B * world,
                   "batches": f"{len(r['batches'])} distinct batches over the same tables "
                              "(table seed = rank), cycled; each step's hot set was learned "
                              "on the batch before",
                   "parallelism": f"replicas x{world} (independent batches)",
                   "l2": f"inputs larger than L2 (indices {w.n * INDEX_BYTES / 1e9:.2f} GB "
                         f"per batch, weights "
                         f"{w.weights.numel() * w.weights.element_size() / 1e9:.1f} GB); no flush",
                   "storage": f"{args.weights} weights, fp32 "
                              f"{'per-element' if ew else 'per-row'} momentum, fp32 gradients"},
        "phases_ms": {"preprocess": r["pre_ms"], "forward": r["fwd_ms"], "update": r["upd_ms"],
                      "note": "median per step; the sort chain runs on a side stream during "
                              "the forward and is waited for by the update"},
        "hot_rows": {"hit_rate": u["hit_rate"], "cold_lookups": u["cold_lookups"],
                     "hot_rows": u["hot_rows_next"],
                     "hit_rate_per_batch": [x["hit_rate"] for x in r["units_per_batch"]],
                     "note": "fraction of lookups served by hot rows learned on the previous "
                             "batch"},
        "cold_start_ms": dict(r["cold_start"], note="one step whose hot set is empty (a "
                                                    "fresh workspace's first batch)"),
        "runs": {k: u[k] for k in ("R", "long_runs", "long_chunks", "short_runs",
                                   "short_pairs", "long_pairs")},
        "roofline": kernels[ROOFLINE_DOMINANT],
        "roofline_kernels": {k: v for k, v in kernels.items() if k != ROOFLINE_DOMINANT},
        "problem_roofline": {
            k: {"min_bytes": cb[k], "ms": t, "GBps": cb[k] / (t / 1e3) / 1e9,
                "frac": cb[k] / (t / 1e3) / 1e9 / hbm}
            for k, t in (("forward", t_fwd), ("backward", t_bwd), ("step", t_step))},
        "clocks": r["clocks"],
        "gpu_launches": r["launches"],
    }
    line["problem_roofline"]["note"] = ("compulsory bytes over time: forward = preprocess + "
                                        "forward phases, backward = update phase")
    if "e2e_ms" in r:
        line["e2e"] = {"value": r["e2e_lookups"] * world / (r["e2e_ms"] / 1e3),
                       "unit": "lookups/s", "h2d_bytes_per_step": r["h2d"],
                       "d2h_bytes_per_step": r["d2h"],
                       "copy_streams": r["e2e_copy_streams"], "link": r["link"]}
    if not args.no_configs and not reduced and world == 1 and args.weights == "fp16" \
            and not ew and args.pooling == "sum":
        import table_embedding_bag_gb300 as tbe
        line["configs"] = measure_configs(tbe, w.indices.device, rank, args, hbm,
                                          main=(r["batches"], r["stepper"]))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        mean, ew_ = args.pooling == "mean", args.optimizer == "elementwise"
        s = cpu_sample(w, args.cpu_bags)
        dt = time_oracle(s, mean, ew_)
        cores = max(1, os.cpu_count() or 1)
        per = max(1, min(args.cpu_bags, w.B // cores))  # bags of table 0 per core
        v, n_all, secs = cpu_baseline_parallel(w, per, cores, mean, ew_)
        line["cpu_baseline"] = {"value": v, "unit": "lookups/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"table 0 of the first batch, {cores} disjoint ranges "
                                          f"of {per} bags ({n_all} lookups), forward + "
                                          f"backward, one oracle process per core, "
                                          f"{secs:.1f} s wall",
                                "single_core": {"value": s.n / dt, "cores": 1,
                                                "sample": f"the first {args.cpu_bags} bags "
                                                          f"({s.n} lookups)"},
                                "openmp": cpu_baseline_openmp(w, per * cores, cores, mean, ew_)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
