"""Every element of the full-size shards against the oracle.

The benchmark's own shard (1,722,408,960 elements, 293 tensors, GAS 4, two
steps) in the benchmark's launch configuration (last micro-batch deferred into
the fused step), with every micro-batch deferred, and with every micro-batch
stored; the 1.83e9-element GAS-32 partition with the last micro-batch
deferred and with all 32 gradients resident; and the 3,700,064,256-element
ragged list of 72 separately allocated tensors (GAS 8, two steps) with the
last micro-batch deferred.  The GPU runs all variants first
and keeps their states resident; the oracle then runs the shard one host
slice at a time (inputs regenerated from the counters, the global clip
coefficient of every step streamed beforehand) and each slice is compared
element by element with every variant: m, v and master within the tolerance,
the bf16 parameters by the bf16 rule, and the stored accumulator bit for bit
after as many micro-batches as the variant stored.
"""
import json

import pytest

torch = pytest.importorskip("torch")

from synth import workloads  # noqa: E402
from harness import GpuShard, check_norms, dense_streamed_parity  # noqa: E402
from mixed_precision_optimizer_bf16_gb300.optimizer import resident_pattern  # noqa: E402

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")


def _run_dense(wl, patterns):
    shards = {}
    try:
        for name, pat in patterns.items():
            sh = GpuShard(wl, defer=pat)
            sh.run(wl.steps)
            shards[name] = sh
        stats, sums = dense_streamed_parity(wl, shards, wl.steps)
        for name, sh in shards.items():
            stats[name]["norm_rel_err"] = check_norms(sh.norms, sums)
    finally:
        for sh in shards.values():
            sh.close()
        shards.clear()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    for name, st in stats.items():
        assert st["elements"] == wl.n
        print("dense", wl.name, name, json.dumps(st))
    return stats


@needs_cuda
def test_scaled_bloom_full_size_dense():
    wl = workloads.workload(2)
    _run_dense(wl, {"last_deferred": True, "all_deferred": [True] * wl.gas, "stored": False})


@needs_cuda
def test_large_partition_full_size_dense():
    wl = workloads.workload(3)
    _run_dense(wl, {"last_deferred": True, "resident_in_eights": resident_pattern(wl.gas)})


@needs_cuda
def test_tp4_slice_full_size_dense():
    wl = workloads.workload(4)
    _run_dense(wl, {"last_deferred": True})
