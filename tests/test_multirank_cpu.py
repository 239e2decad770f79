"""The benchmark's multi-rank path on CPU (gloo, world size 2).

With N > 1 every rank runs an independent replica of the shard (no data-path
collective); the job time is the maximum over ranks, rank 0 alone prints, and
under --impl reference only rank 0 runs the CPU oracle.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
    buf = io.StringIO()
    with redirect_stdout(buf):
        args = type("A", (), dict(steps=1, warmup=0, workload=1))()
        if rank != 0:
            bench.run_reference(args)   # non-zero ranks do no work and print nothing
    dist.barrier()
    q.put((rank, got, buf.getvalue(), bench.rank_info()))
    dist.destroy_process_group()


def test_max_over_ranks_and_rank0_only_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]          # both ranks see the slowest rank's time
    assert res[1][2] == ""                               # rank 1 printed nothing
    assert res[0][3] == (0, 2, 0) and res[1][3] == (1, 2, 1)


def _gather_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    from mixed_precision_optimizer_bf16_gb300 import bf16opt as C
    from mixed_precision_optimizer_bf16_gb300.optimizer import gather_sumsqs
    # values whose sum depends on the order: rank order must be used on every rank
    local = [1.0, 1e-16, -1.0][rank]
    parts = gather_sumsqs(local)
    rc, total = C.bf16opt_sum_rank_sumsqs(parts)
    q.put((rank, parts, rc, total))
    dist.destroy_process_group()


def test_global_sumsq_rank_order_gloo():
    """Each rank's local sum of squares is all-gathered in rank order and the
    library sums the gathered values in that order, so every rank clips with
    the same bits."""
    world = 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = (1.0 + 1e-16) + -1.0          # = 0.0 in rank order (1 + 1e-16 rounds to 1)
    assert want == 0.0 and (1.0 + (1e-16 + -1.0)) != 0.0
    assert [r[1] for r in res] == [[1.0, 1e-16, -1.0]] * world
    assert [(r[2], r[3]) for r in res] == [(0, want)] * world


def test_max_over_ranks_without_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5


def test_reference_arm_under_torchrun():
    """The driver's launch of the reference arm for N > 1: torchrun, two ranks;
    rank 0 alone times the oracle and prints exactly one JSON line, the other
    rank exits 0 without work."""
    import json
    import subprocess

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(root, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
