"""TBE training-step benchmark: pooled forward + backward with row-wise Adagrad.

One step = tbe_forward (pooled lookup) + tbe_preprocess (expand, radix sort,
run-length encode, classify) + tbe_backward_rowwise_adagrad on the
preprocessed runs (short-run and long-run update kernels), over one batch of
the hot-row workload: T=8 tables of E=1e7 rows, D=128, fp16 weights (20.5 GB)
+ fp32 row-wise momentum, B=131072 bags per table, L=200 lookups per bag
(209.7M lookups), Zipf(1.4) rows over a per-table random permutation.  Inputs
are drawn on the device once (seeded) and stay resident; every timed step
applies a real optimizer update.  Indices (1.7 GB) and weights (20.5 GB) are
far larger than the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Rank 0 prints one JSON line.  With N > 1 (torchrun) every rank runs its own
independent batch (different seed): weak scaling with no collective on the
data path; value = lookups of all ranks / max-over-ranks time.
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
    p.add_argument("--pooling", choices=["sum", "mean"], default="sum",
                   help="pooling mode of the step (the recorded workload is sum)")
    p.add_argument("--weights", choices=["fp16", "bf16"], default="fp16",
                   help="weight type (the recorded workload is fp16)")
    p.add_argument("--optimizer", choices=["rowwise", "elementwise"], default="rowwise",
                   help="Adagrad form (the recorded workload is row-wise)")
    # smaller variants of the hot-row recipe, for profiling captures only
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


# The step's dominant kernel (largest share of the ncu launch list of this
# workload, profiles/launches_hot_row_step.md): the long-run chunk kernel of
# the backward.  Its launches are timed live by the library's kernel probe.
ROOFLINE_KERNEL = "long_chunks_kernel (tbe_backward_rowwise_adagrad, long runs)"
ROOFLINE_KERNEL_SOURCES = ("update.cu", "common.cuh")
ROOFLINE_PROFILE = "long_chunks_hot_row.md"


def source_sha1():
    """First 16 hex digits of the sha1 over the roofline kernel's sources."""
    import hashlib
    h = hashlib.sha1()
    for f in ROOFLINE_KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "table_embedding_bag_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes of one launch of the roofline kernel on this workload, from
    the committed ncu summary, if the kernel's sources are unchanged since
    the capture (else None)."""
    path = os.path.join(ROOT, "profiles", ROOFLINE_PROFILE)
    try:
        text = open(path).read()
        digest = source_sha1()
    except OSError:
        return None
    fields = dict(line.split(":", 1) for line in text.splitlines()
                  if line.startswith(("traffic_bytes_per_launch:", "source_sha1:")))
    if fields.get("source_sha1", "").strip() != digest:
        return None
    return int(fields["traffic_bytes_per_launch"])


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


def long_chunk_bytes(D, long_pairs, chunks, long_runs, elementwise=False):
    """Algorithmic bytes of one long_chunks_kernel launch, counted per use (the
    per-unit figures of the design notes): per long pair its gradient row
    (4 D) and pair data (8); per chunk its partial written and read back
    (2 x 4 D) and its descriptor (16); per long run the weights row read and
    written (2 x 2 D), the momentum (8, or 8 D element-wise) and the run
    record (32)."""
    return (long_pairs * (4 * D + 8) + chunks * (2 * 4 * D + 16)
            + long_runs * (2 * 2 * D + momentum_bytes(D, elementwise) + 32))


def forward_problem_bytes(w, rows_touched):
    """Compulsory bytes of the forward problem: indices, offsets, every
    distinct row once, the pooled output."""
    nb = w.T * w.B
    D = int(w.D[0])
    return (w.n * INDEX_BYTES + (nb + 1) * INDEX_BYTES + rows_touched * D * 2
            + w.B * int(w.D.sum()) * 4)


def problem_roofline(w, rows_touched, r, peak, elementwise=False):
    """Compulsory bytes of the forward, the backward and the whole step (each
    index and offset read once, every distinct row once, the output written
    once, grad_out read once, each touched row's weights and momentum read and
    written once) over their measured time, against the HBM peak.  The
    preprocess reads the indices for both passes, so its time counts in both."""
    nb = w.T * w.B
    D = int(w.D[0])
    idx = w.n * INDEX_BYTES + (nb + 1) * INDEX_BYTES
    out = w.B * int(w.D.sum()) * 4
    fwd = idx + rows_touched * D * 2 + out
    upd = rows_touched * (4 * D + momentum_bytes(D, elementwise))
    bwd = idx + out + upd  # grad_out has the output's size
    step = idx + 2 * out + upd
    t = {"forward": r["pre_ms"] + r["fwd_ms"], "backward": r["pre_ms"] + r["upd_ms"],
         "step": r["ms"] / r["steps"]}
    res = {}
    for k, b in (("forward", fwd), ("backward", bwd), ("step", step)):
        gbs = b / (t[k] / 1e3) / 1e9
        res[k] = {"min_bytes": b, "ms": t[k], "GBps": gbs, "frac": gbs / peak}
    res["note"] = "compulsory bytes over time; preprocess time counted in forward and backward"
    return res


def run_native(args, world, rank, local):
    import table_embedding_bag_gb300 as tbe
    import workloads

    dev = torch.device("cuda", torch.cuda.current_device())
    E_scale = None if args.rows is None else args.rows / workloads.SPECS["hot"].E
    wdt = torch.bfloat16 if args.weights == "bf16" else torch.float16
    w = workloads.make("hot", device=dev, seed=rank, T=args.tables, B=args.bags, E_scale=E_scale,
                       weights_dtype=wdt)
    desc = tbe.TBEDesc(w.E, w.D, w.B, w.indices.dtype, dev, wdt)
    mean = args.pooling == "mean"
    ew = args.optimizer == "elementwise"
    ws = tbe.Workspace(desc, w.n, False, dev, mean=mean)
    weights = w.weights
    momentum = (torch.zeros(desc.num_weights, dtype=torch.float32, device=dev) if ew
                else w.momentum)
    out = torch.empty(w.B, desc.total_D, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    PRE = tbe.TBE_F_PREPROCESSED | (tbe.TBE_F_MEAN if mean else 0)
    UPD = PRE | (tbe.TBE_F_ELEMENTWISE if ew else 0)

    def step(ev=None):
        # one preprocess of the batch's indices serves forward and backward
        if ev is not None:
            ev[0].record(stream)
        tbe.tbe_preprocess(desc, w.indices, w.offsets, None, ws)
        if ev is not None:
            ev[1].record(stream)
        tbe.tbe_forward(desc, weights, w.indices, w.offsets, None, out, ws, PRE)
        if ev is not None:
            ev[2].record(stream)
        tbe.tbe_backward_rowwise_adagrad(desc, w.grad_out, w.indices, w.offsets, None, weights,
                                         momentum, w.lr, w.eps, ws, UPD)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = Clocks(local)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    tbe.tbe_probe_set(tbe.TBE_PROBE_LONG_CHUNKS)
    launches0 = tbe.tbe_kernel_launches()
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    launches = tbe.tbe_kernel_launches() - launches0
    probe_launches, probe_ms = tbe.tbe_probe_read()
    tbe.tbe_probe_set(tbe.TBE_PROBE_OFF)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    status = tbe.tbe_read_status(ws)
    if status & tbe.TBE_ERR_TIMEOUT:
        raise SystemExit("bench: a kernel's bounded wait timed out during the timed steps "
                         f"(status {status:#x}); the measurement is invalid")
    ms_local = t0.elapsed_time(t1)
    ms = max_over_ranks(ms_local, world, dev)
    pre = [e[0].elapsed_time(e[1]) for e in evs]
    fwd = [e[1].elapsed_time(e[2]) for e in evs]
    upd = [e[2].elapsed_time(e[3]) for e in evs]

    view = tbe.tbe_workspace_view(desc, w.n, ws)
    off = view["counts"] - ws.buf.data_ptr()
    counts = ws.buf[off:off + 32].view(torch.int32).cpu().numpy().view(np.uint32)
    R, n_long, n_chunks = int(counts[0]), int(counts[2]), int(counts[3])
    n_cold = int(counts[7])  # lookups left to the sort after the hot rows
    # hot rows per table (the set the next step uses; the same batch repeats,
    # so it is also the set the timed steps used)
    hoff = view["hot_n"] - ws.buf.data_ptr()
    n_hot = int(ws.buf[hoff:hoff + 4 * w.T].view(torch.int32).cpu().numpy().sum())

    def ws_u32(ptr, count):
        o = ptr - ws.buf.data_ptr()
        return ws.buf[o:o + 4 * count].view(torch.int32).cpu().numpy().view(np.uint32)

    # pairs of the long runs (the units of the long-run kernel)
    run_pairs = ws_u32(view["run_pairs"], R + 1).astype(np.int64)
    long_idx = ws_u32(view["long_runs"], n_long).astype(np.int64)
    long_pairs = int((run_pairs[long_idx + 1] - run_pairs[long_idx]).sum()) if n_long else 0
    result = {
        "ms": ms, "ms_local": ms_local, "fwd_ms": statistics.median(fwd),
        "pre_ms": statistics.median(pre), "upd_ms": statistics.median(upd),
        "n": w.n, "R": R, "n_long": n_long, "n_chunks": n_chunks, "n_cold": n_cold,
        "n_hot": n_hot, "long_pairs": long_pairs, "clocks": clk,
        "probe_launches": probe_launches, "probe_ms": probe_ms,
        "launches": launches, "w": w,
    }

    if not args.no_e2e:
        # End to end through the public API: per step, this step's inputs go
        # host -> device from pinned memory and the pooled output comes back.
        # Two device input slots: step k+1's uploads (copy stream) overlap
        # step k's compute, and step k's output download (a third stream)
        # overlaps its backward; every copy stays inside the timed region.
        h_idx = w.indices.cpu().pin_memory()
        h_off = w.offsets.cpu().pin_memory()
        h_grad = w.grad_out.cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        slots = [(torch.empty_like(w.indices), torch.empty_like(w.offsets),
                  torch.empty_like(w.grad_out)) for _ in range(2)]
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        copied = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        fwd_done, out_read = torch.cuda.Event(), torch.cuda.Event()

        def e2e_step(k):
            d_idx, d_off, d_grad = slots[k % 2]
            with torch.cuda.stream(up):
                if k >= 2:
                    up.wait_event(consumed[k % 2])
                d_idx.copy_(h_idx, non_blocking=True)
                d_off.copy_(h_off, non_blocking=True)
                d_grad.copy_(h_grad, non_blocking=True)
                copied[k % 2].record(up)
            stream.wait_event(copied[k % 2])
            if k >= 1:
                stream.wait_event(out_read)  # the previous output was read back
            tbe.tbe_preprocess(desc, d_idx, d_off, None, ws)
            tbe.tbe_forward(desc, weights, d_idx, d_off, None, out, ws, PRE)
            fwd_done.record(stream)
            with torch.cuda.stream(down):
                down.wait_event(fwd_done)
                h_out.copy_(out, non_blocking=True)
                out_read.record(down)
            tbe.tbe_backward_rowwise_adagrad(desc, d_grad, d_idx, d_off, None, weights, momentum,
                                             w.lr, w.eps, ws, UPD)
            consumed[k % 2].record(stream)

        for k in range(max(1, args.warmup)):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier(world)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        up.wait_event(a)
        down.wait_event(a)
        for k in range(args.steps):
            e2e_step(k + 2 * args.warmup)  # the slot pattern continues past the warm-up
        stream.wait_event(out_read)
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(a.elapsed_time(b), world, dev)
        result["e2e_ms"] = e2e_ms
        result["h2d"] = h_idx.numel() * h_idx.element_size() + h_off.numel() * 8 + \
            h_grad.numel() * 4
        result["d2h"] = h_out.numel() * 4
    return result


def cpu_sample(w_dev, bags):
    """Table 0, its first `bags` bags, as a standalone host problem holding
    only the rows those bags touch (renumbered)."""
    import workloads
    off = w_dev.offsets[:bags + 1].cpu().numpy()
    idx_dev = w_dev.indices[:int(off[-1])]
    uniq, inv = torch.unique(idx_dev, return_inverse=True)
    D0 = int(w_dev.D[0])
    rows = w_dev.weights[:int(w_dev.E[0]) * D0].view(-1, D0)[uniq].cpu().reshape(-1)
    if rows.dtype != torch.bfloat16:
        rows = rows.numpy()
    G0 = w_dev.grad_out[:bags, :D0].cpu().numpy()
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
    W = s.weights.view(torch.int16).numpy().view(np.uint16) if bf16 else s.weights.numpy()
    G = s.grad_out.numpy()
    m = (np.zeros(int(tab.w_offsets[-1]), np.float32) if elementwise
         else s.momentum.numpy())
    t = time.perf_counter()
    oracle.forward(tab, s.B, W, idx, off, mean=mean, bf16=bf16)
    oracle.backward_rowwise_adagrad(tab, s.B, idx, off, G, W, m, s.lr, s.eps, mean=mean,
                                    bf16=bf16, elementwise=elementwise)
    return time.perf_counter() - t


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
        bags = 2048
        times, lookups = [], 0
        for k in range(args.warmup + args.steps):
            s = reference_sample(bags, seed=k, weights_dtype=torch.bfloat16
                                 if args.weights == "bf16" else torch.float16)
            dt = time_oracle(s, args.pooling == "mean", args.optimizer == "elementwise")
            if k >= args.warmup:
                times.append(dt)
                lookups += s.n
        tot = sum(times)
        value = lookups / tot
        line = {
            "impl": "reference", "metric": METRIC, "value": value, "unit": "lookups/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(args), "sample": f"table 0, {bags} bags x 200 lookups "
                                                     "per step (same recipe, host-drawn, "
                                                     "touched rows only)"},
            "cpu_baseline": {"value": value, "unit": "lookups/s", "cores": 1, "kind": "oracle",
                             "sample": f"table 0 of the hot-row recipe, {bags} bags x 200 "
                                       "lookups per step, forward + backward"},
            "e2e": {"value": value, "unit": "lookups/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return

    r = run_native(args, world, rank, local)
    w = r["w"]
    total_lookups = w.n * world * args.steps
    value = total_lookups / (r["ms"] / 1e3)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    D = int(w.D[0])
    ew = args.optimizer == "elementwise"
    kb = long_chunk_bytes(D, r["long_pairs"], r["n_chunks"], r["n_long"], ew)
    k_launch_ms = r["probe_ms"] / max(r["probe_launches"], 1)
    achieved = kb / (k_launch_ms / 1e3) / 1e9
    fwd_problem = forward_problem_bytes(w, r["R"] + r["n_hot"])
    line = {
        "metric": METRIC, "value": value, "unit": "lookups/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_name(
                       args, WORKLOAD if (args.tables, args.rows, args.bags) == (None,) * 3
                       else f"reduced hot-row recipe T={w.T} E={int(w.E[0])} B={w.B} "
                            "(profiling case)"),
                   "n_lookups": w.n, "global_batch": w.B * world,
                   "parallelism": f"replicas x{world} (independent batches)",
                   "l2": f"inputs larger than L2 (indices {w.n * INDEX_BYTES / 1e9:.2f} GB, "
                         f"weights {w.weights.numel() * 2 / 1e9:.1f} GB); no flush",
                   "storage": f"{args.weights} weights, fp32 "
                              f"{'per-element' if ew else 'per-row'} momentum, fp32 gradients"},
        "phases_ms": {"forward": r["fwd_ms"], "preprocess": r["pre_ms"], "update": r["upd_ms"]},
        "runs": {"R": r["R"], "long_runs": r["n_long"], "long_chunks": r["n_chunks"],
                 "cold_lookups": r["n_cold"], "hot_rows": r["n_hot"]},
        "roofline": {"kernel": ROOFLINE_KERNEL, "bound": "hbm", "achieved": achieved,
                     "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": profiled_traffic() if args.tables is None else None,
                     "peak_source": peak_src,
                     "bytes_model": "per use: gradient row + pair data per long pair, "
                                    "partial write+read per chunk, weights row r/w + "
                                    "momentum per long run",
                     "bytes_per_launch": kb, "launch_ms": k_launch_ms,
                     "launches_timed": r["probe_launches"],
                     "units": {"long_pairs": r["long_pairs"], "chunks": r["n_chunks"],
                               "long_runs": r["n_long"]}},
        "forward_context": {"phase_ms": r["fwd_ms"],
                            "problem_min_GBps": fwd_problem / (r["fwd_ms"] / 1e3) / 1e9},
        "problem_roofline": problem_roofline(w, r["R"] + r["n_hot"], dict(r, steps=args.steps), hbm,
                                             ew),
        "clocks": r["clocks"],
        "gpu_launches": r["launches"],
    }
    if "e2e_ms" in r:
        line["e2e"] = {"value": total_lookups / (r["e2e_ms"] / 1e3), "unit": "lookups/s",
                       "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = cpu_sample(w, args.cpu_bags)
        dt = time_oracle(s, args.pooling == "mean", args.optimizer == "elementwise")
        line["cpu_baseline"] = {"value": s.n / dt, "unit": "lookups/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"table 0, first {args.cpu_bags} bags "
                                          f"({s.n} lookups), forward + backward"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
