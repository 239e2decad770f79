"""ZeRO-Offload variant (bf16opt_create_offload): FP32 master and moments in
host memory, updated by the host cores; accumulator, norm and bf16
parameters on the GPU.

The host update repeats the device step's FP32 operations with the scalars
and clip coefficient the device computed, so an offload handle and a device
handle fed the same gradients hold the same bits after every step; both equal
the oracle within the tolerance.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth import gpu as sgpu, workloads  # noqa: E402
from harness import GpuShard, check_norms, compare, oracle_dense  # noqa: E402
from mixed_precision_optimizer_bf16_gb300 import bf16opt as C  # noqa: E402
from mixed_precision_optimizer_bf16_gb300.optimizer import BF16Optimizer  # noqa: E402

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")


class OffloadShard:
    """A FLAT workload with its master and moments in host memory."""

    def __init__(self, wl, pattern, threads=0):
        self.wl, self.pattern = wl, pattern
        dev = torch.empty(wl.n + wl.misalign + 64, dtype=torch.float32, device="cuda")
        master = torch.empty(wl.n, dtype=torch.float32, device="cuda")
        sgpu.fill_master(wl, master)
        self.state = dict(master=master.cpu(), exp_avg=torch.zeros(wl.n, dtype=torch.float32),
                          exp_avg_sq=torch.zeros(wl.n, dtype=torch.float32),
                          grad_accum=dev[wl.misalign:wl.misalign + wl.n],
                          param_bf16=torch.empty(wl.n + wl.misalign + 64, dtype=torch.int16,
                                                 device="cuda")[wl.misalign:wl.misalign + wl.n])
        self.opt = BF16Optimizer(wl.groups, flat=self.state, ranges=wl.ranges(), max_grad_norm=wl.max_norm,
                                 offload=True, offload_threads=threads)
        nbuf = wl.gas if any(pattern[:-1]) else 1
        self.gbufs = [torch.empty(wl.n + wl.misalign + 64, dtype=torch.int16,
                                  device="cuda")[wl.misalign:wl.misalign + wl.n] for _ in range(nbuf)]
        self.norms = []

    def run(self, steps, lr=None):
        for s in range(steps):
            for k in range(self.wl.gas):
                buf = self.gbufs[k % len(self.gbufs)]
                sgpu.fill_grad(self.wl, s, k, buf)
                self.opt.accumulate(buf, first=k == 0, last=k == self.wl.gas - 1, defer=self.pattern[k])
            self.norms.append(self.opt.grad_norm(sync=True))
            self.opt.step(lr=lr)
        torch.cuda.synchronize()

    def states(self):
        return dict(p=self.state["master"].numpy().copy(), m=self.state["exp_avg"].numpy().copy(),
                    v=self.state["exp_avg_sq"].numpy().copy(), acc=self.state["grad_accum"].cpu().numpy(),
                    p_bf16=self.state["param_bf16"].cpu().numpy().view(np.uint16))


def _same_bits(a, b, keys=("p", "m", "v", "p_bf16")):
    for k in keys:
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k


@needs_cuda
@pytest.mark.parametrize("pattern", [[False, False, True], [True, True, True], [False, False, False]])
def test_offload_equals_device_step_and_oracle(pattern):
    wl = workloads.custom(970, [60_001, 333, 20_000], decay=[True, False, True], gas=3, steps=3, grad_sigma=0.3,
                          misalign=1)
    off = OffloadShard(wl, pattern, threads=3)
    off.run(wl.steps)
    got = off.states()
    dev = GpuShard(wl, defer=pattern)
    dev.run(wl.steps)
    want = dev.states()
    assert off.norms == dev.norms and off.opt.t == dev.opt.t == wl.steps
    dev.close()
    off.opt.close()
    _same_bits(got, want)
    ref, scales = oracle_dense(wl, wl.steps)
    check_norms(off.norms, ref["sumsq"])
    # the offloaded step folds deferred micro-batches into the stored accumulator first
    compare(got, ref, scales, wl, check_acc=True)


@needs_cuda
def test_offload_blocks_and_schedule():
    """2^25 + 12,345 elements: three pipelined blocks of 2^24 and a ragged one;
    an LR schedule and a per-step learning-rate override; the default thread
    count.  Bit-identical to the device step."""
    wl = workloads.custom(971, [(1 << 25) + 2345, 10_000], decay=[True, False], gas=2, steps=2, grad_sigma=0.01,
                          misalign=2)
    pattern = [False, True]
    off = OffloadShard(wl, pattern)
    off.opt.set_lr_schedule(1, 4, 0.25)
    off.run(1)
    dev = GpuShard(wl, defer=pattern)
    dev.opt.set_lr_schedule(1, 4, 0.25)
    dev.run_step(0)
    # second step with an override on both
    for sh in (off, dev):
        for k in range(wl.gas):
            buf = sh.gbufs[k % len(sh.gbufs)]
            sgpu.fill_grad(wl, 1, k, buf)
            sh.opt.accumulate(buf, first=k == 0, last=k == wl.gas - 1, defer=pattern[k])
        sh.opt.grad_norm(sync=True)
        sh.opt.step(lr=[3e-5, 1e-4])
    torch.cuda.synchronize()
    _same_bits(off.states(), dev.states())
    dev.close()
    off.opt.close()


@needs_cuda
def test_offload_skips_a_nonfinite_step_and_rejects_wrong_memory():
    wl = workloads.custom(972, [5000], gas=1, steps=1, grad_sigma=0.1)
    off = OffloadShard(wl, [False])
    off.opt.set_skip_nonfinite(True)
    before = off.states()
    g = torch.zeros(wl.n, dtype=torch.float32, device="cuda")
    g[17] = float("inf")
    off.opt.accumulate(g.to(torch.bfloat16).view(torch.int16), first=True, last=True)
    off.opt.grad_norm()
    off.opt.step()
    torch.cuda.synchronize()
    _same_bits(off.states(), before)
    assert off.opt.t == 0
    off.opt.close()
    # master on the device, accumulator on the host: refused
    n = 1000
    d = dict(master=torch.zeros(n, device="cuda"), exp_avg=torch.zeros(n), exp_avg_sq=torch.zeros(n),
             grad_accum=torch.zeros(n, device="cuda"), param_bf16=torch.zeros(n, dtype=torch.int16, device="cuda"))
    desc = C.flat_desc(n, *(d[k].data_ptr() for k in ("master", "exp_avg", "exp_avg_sq", "grad_accum",
                                                       "param_bf16")), wl.groups)
    assert C.bf16opt_create_offload(desc)[0] == C.BF16OPT_ERR_INVALID_ARG
    assert "host memory" in C.bf16opt_last_error(None)
    d["master"], d["grad_accum"] = torch.zeros(n), torch.zeros(n)
    desc = C.flat_desc(n, *(d[k].data_ptr() for k in ("master", "exp_avg", "exp_avg_sq", "grad_accum",
                                                       "param_bf16")), wl.groups)
    assert C.bf16opt_create_offload(desc)[0] == C.BF16OPT_ERR_INVALID_ARG
    assert "current device" in C.bf16opt_last_error(None)


@needs_cuda
def test_offload_checkpoint_resume():
    """state_dict / load_state_dict of an offload optimizer (host master and
    moments, device bf16 parameters): dump after one step, restore into fresh
    buffers, continue -- the same bits as an uninterrupted run."""
    wl = workloads.custom(973, [30_001, 999], decay=[True, False], gas=2, steps=3, grad_sigma=0.2)
    pattern = [False, True]
    full = OffloadShard(wl, pattern)
    full.run(wl.steps)
    want = full.states()
    full.opt.close()

    a = OffloadShard(wl, pattern)
    a.run(1)
    sd = a.opt.state_dict()
    a.opt.close()
    b = OffloadShard(wl, pattern)
    b.opt.load_state_dict(sd)
    for s in range(1, wl.steps):
        for k in range(wl.gas):
            buf = b.gbufs[k % len(b.gbufs)]
            sgpu.fill_grad(wl, s, k, buf)
            b.opt.accumulate(buf, first=k == 0, last=k == wl.gas - 1, defer=pattern[k])
        b.opt.grad_norm()
        b.opt.step()
    torch.cuda.synchronize()
    assert b.opt.t == wl.steps
    _same_bits(b.states(), want)
    b.opt.close()


@needs_cuda
def test_reduce_scatter_without_a_process_group():
    """accumulate_reduce_scatter with no process group initialised: one rank,
    the whole buffer is its partition, the same as plain accumulate calls."""
    wl = workloads.custom(974, [20_000, 77], decay=[True, False], gas=3, steps=2, grad_sigma=0.1)
    dev = GpuShard(wl, defer=[False, False, True])
    dev.run(wl.steps)
    want = dev.states()
    dev.close()
    sh = GpuShard(wl, defer=False)
    for s in range(wl.steps):
        for k in range(wl.gas):
            sgpu.fill_grad(wl, s, k, sh.gbuf)
            sh.opt.accumulate_reduce_scatter(sh.gbuf, first=k == 0, last=k == wl.gas - 1)
        sh.opt.grad_norm_distributed()
        sh.opt.step()
    torch.cuda.synchronize()
    _same_bits(sh.states(), want)
    sh.close()
