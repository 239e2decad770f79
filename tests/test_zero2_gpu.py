"""ZeRO-2 gradient reduction feeding the FP32 accumulation on the GPU.

Three processes stand for three data-parallel ranks; they share cuda:0 and
exchange over gloo (host memory), so no kernel of one process waits on
another's.  Each owns one partition of a flat shard (BF16Optimizer over its
slice); per micro-batch it produces a bf16 gradient of the whole buffer,
accumulate_reduce_scatter exchanges the partitions and folds the received
slices into the FP32 accumulator in rank order through the library (deferred
in runs, the last micro-batch's slices folded by the norm pass and the step),
grad_norm_distributed gives the global norm, and the step runs per partition.
Put together the partitions equal the oracle on the whole shard with the
world x GAS gradients as micro-batches in (micro-batch, rank) order.
"""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD, GAS = 3, 3


def _workload():
    from synth import workloads
    return workloads.custom(961, [40_001, 777, 19_000], decay=[True, False, True], gas=GAS * WORLD, steps=2,
                            grad_sigma=0.3, misalign=1)


def _worker(rank, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=WORLD)
    try:
        torch.cuda.set_device(0)
        from synth import gpu as sgpu
        from mixed_precision_optimizer_bf16_gb300.optimizer import BF16Optimizer, alloc_flat, partition_bounds
        wl = _workload()
        b = partition_bounds(wl.n, WORLD)
        lo, hi = b[rank], b[rank + 1]
        st = alloc_flat(hi - lo, "cuda", wl.misalign)
        sgpu.fill_master(wl, st["master"], lo)
        for k in ("exp_avg", "exp_avg_sq", "grad_accum", "param_bf16"):
            st[k].zero_()
        rg = [(max(x, lo) - lo, min(y, hi) - lo, gi) for x, y, gi in wl.ranges() if max(x, lo) < min(y, hi)]
        opt = BF16Optimizer(wl.groups, flat=st, ranges=rg, max_grad_norm=wl.max_norm)
        full = torch.empty(wl.n + 64, dtype=torch.int16, device="cuda")[wl.misalign:wl.misalign + wl.n]
        norms = []
        for s in range(wl.steps):
            for k in range(GAS):
                sgpu.fill_grad(wl, s, k * WORLD + rank, full)
                opt.accumulate_reduce_scatter(full, first=k == 0, last=k == GAS - 1)
            norms.append(opt.grad_norm_distributed())
            opt.step()
        torch.cuda.synchronize()
        out = {k: st[n].cpu().numpy() for k, n in (("p", "master"), ("m", "exp_avg"), ("v", "exp_avg_sq"),
                                                   ("acc", "grad_accum"))}
        out["p_bf16"] = st["param_bf16"].cpu().numpy().view(np.uint16)
        opt.close()
        q.put((rank, out, norms))
    finally:
        dist.destroy_process_group()


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_zero2_reduce_scatter_feeds_the_fp32_accumulator():
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from harness import check_norms, compare, oracle_dense
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=600) for _ in range(WORLD)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    wl = _workload()
    ref, scales = oracle_dense(wl, wl.steps)
    for r in res:
        assert r[2] == res[0][2]                  # every rank clips with the same norm
    check_norms(res[0][2], ref["sumsq"])
    got = {k: np.concatenate([r[1][k] for r in res]) for k in ("p", "m", "v", "p_bf16", "acc")}
    # the stored accumulator holds every micro-batch but the last one's slices (deferred into the step)
    last_stored = np.empty(wl.n, np.float32)
    import oracle
    import synth
    for j in range((GAS - 1) * WORLD):
        oracle.accumulate(last_stored, synth.fill_grad(wl, wl.steps - 1, j, np.empty(wl.n, np.uint16)), first=j == 0)
    compare(got, ref, scales, wl, check_acc=last_stored)
