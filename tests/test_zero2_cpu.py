"""ZeRO-2 gradient reduction feeding the FP32 accumulation, on CPU (gloo, 3 ranks).

Every rank holds a bf16 gradient of the whole flat buffer per micro-batch; the
partitions are exchanged (optimizer.exchange_gradient_slices) and each owner
folds the received slices of its partition in rank order.  Here the owner's
fold, norm and AdamW are the oracle's, so the test checks the exchange and its
ordering without a GPU: put together, the partitions must equal the oracle run
on the whole shard with the world x GAS gradients as micro-batches in
(micro-batch, rank) order -- the accumulator bit for bit.
"""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD, GAS = 3, 2


def _workload():
    from synth import workloads
    # micro-batch j = k * WORLD + r is rank r's gradient of micro-batch k
    return workloads.custom(960, [20_011, 333, 9_000], decay=[True, False, True], gas=GAS * WORLD, steps=2,
                            grad_sigma=0.3, zero_frac=0.02)


def _worker(rank, port, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=WORLD)
    try:
        import oracle
        import synth
        from harness import ogroups
        from mixed_precision_optimizer_bf16_gb300 import bf16opt as C
        from mixed_precision_optimizer_bf16_gb300.optimizer import (exchange_gradient_slices, gather_sumsqs,
                                                                    partition_bounds)
        wl = _workload()
        b = partition_bounds(wl.n, WORLD)
        lo, hi = b[rank], b[rank + 1]
        p = synth.fill_master(wl, np.empty(hi - lo, np.float32), lo)
        m, v = np.zeros(hi - lo, np.float32), np.zeros(hi - lo, np.float32)
        pb = oracle.f32_to_bf16(p)
        acc = np.empty(hi - lo, np.float32)
        G = ogroups(wl)
        rg = [(max(x, lo) - lo, min(y, hi) - lo, gi) for x, y, gi in wl.ranges() if max(x, lo) < min(y, hi)]
        sums = []
        for s in range(wl.steps):
            for k in range(GAS):
                full = synth.fill_grad(wl, s, k * WORLD + rank, np.empty(wl.n, np.uint16))
                ph = (7 * s + 3 * k + rank) % 32          # any row phase gives the same rows
                recv = exchange_gradient_slices(torch.from_numpy(full.view(np.int16)), b, phase=ph)
                assert tuple(recv.shape) == (WORLD, hi - lo)
                assert all((recv[q].data_ptr() // 2) % 32 == ph for q in range(WORLD))
                for src in range(WORLD):
                    want = synth.fill_grad(wl, s, k * WORLD + src, np.empty(hi - lo, np.uint16), lo)
                    got = recv[src].numpy().view(np.uint16)
                    assert np.array_equal(got, want), (rank, src)
                    oracle.accumulate(acc, got.copy(), first=k == 0 and src == 0)
            parts = gather_sumsqs(oracle.sumsq(acc))
            rc, total = C.bf16opt_sum_rank_sumsqs(parts)
            assert rc == 0
            sums.append(total)
            c = oracle.clip_coef(total, wl.max_norm)
            for x, y, gi in rg:
                oracle.adamw(p[x:y], m[x:y], v[x:y], pb[x:y], acc[x:y], c, G[gi], s + 1)
        q.put((rank, dict(p=p, m=m, v=v, p_bf16=pb, acc=acc), sums))
    finally:
        dist.destroy_process_group()


def test_zero2_exchange_and_rank_ordered_fold_gloo():
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from harness import compare, oracle_dense
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in range(WORLD)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl = _workload()
    got = {k: np.concatenate([r[1][k] for r in res]) for k in ("p", "m", "v", "p_bf16", "acc")}
    ref, scales = oracle_dense(wl, wl.steps)
    for r in res:    # every rank has the same global sums of squares
        assert r[2] == res[0][2]
        for S, S_ref in zip(r[2], ref["sumsq"]):
            assert abs(S - S_ref) <= 1e-14 * S_ref
    compare(got, ref, scales, wl)    # accumulator bit for bit, states within the tolerance


@pytest.mark.parametrize("world", [1, 2, 3, 7, 8, 9, 16, 17])
@pytest.mark.parametrize("last", [False, True])
def test_fold_pattern_keeps_the_library_limits(world, last):
    """The received slices ride on DEFER: never more than 8 pending (the
    library's limit), a non-last micro-batch folds all of its slices by its
    final one (so the receive buffer can be reused), and the last micro-batch
    leaves at most 8 deferred into the norm pass and the step."""
    from mixed_precision_optimizer_bf16_gb300.optimizer import fold_pattern
    flags = fold_pattern(world, last)
    assert len(flags) == world
    pending = 0
    for f in flags:
        pending = pending + 1 if f else 0
        assert pending <= 8
    if not last:
        assert flags[-1] is False
    else:
        assert flags[-1] is True and pending == (world % 8 or 8) if world > 8 else all(flags)


def test_partition_bounds():
    from mixed_precision_optimizer_bf16_gb300.optimizer import partition_bounds
    assert partition_bounds(10, 3) == [0, 4, 8, 10]
    assert partition_bounds(12, 4) == [0, 3, 6, 9, 12]
    assert partition_bounds(5, 8) == [0, 1, 2, 3, 4, 5, 5, 5, 5]
    for n, w in ((1_722_408_960, 8), (7, 7), (1, 1)):
        b = partition_bounds(n, w)
        assert b[0] == 0 and b[-1] == n and all(x <= y for x, y in zip(b, b[1:]))
