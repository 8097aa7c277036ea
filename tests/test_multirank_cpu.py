"""The multi-process launch path of bench.py on CPU: world size 2 over gloo.
Ranks run independent batches and meet only for the barrier and the
max-over-ranks time; under torchrun the reference arm runs on rank 0 alone."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _max_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(world)
    q.put((rank, bench.max_over_ranks(10.0 + rank, world, torch.device("cpu"))))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in procs)
    assert got == [(0, 11.0), (1, 11.0)]


def test_reference_arm_under_torchrun_prints_one_line():
    port = 29600 + os.getpid() % 1000
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("variant,words", [
    (["--weights", "bf16"], ["bf16 weights", "row-wise momentum"]),
    (["--optimizer", "elementwise"], ["fp16 weights", "per-element momentum"]),
    (["--pooling", "mean"], ["fp16 weights", "mean pooling"]),
])
def test_reference_arm_names_the_variant_it_timed(variant, words):
    # the oracle sample follows the step's options, and the line says which
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
           *variant]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["value"] > 0
    for w in words:
        assert w in line["config"]["workload"]
