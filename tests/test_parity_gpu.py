"""GPU parity: libbf16opt.so (through its C ABI) against the CPU oracle.

Every test here needs a CUDA GPU and the built library; all are marked gpu.
"""
import ctypes
import math
import gc

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402
from synth import gpu as sgpu, workloads  # noqa: E402
from mixed_precision_optimizer_bf16_gb300 import bf16opt as C  # noqa: E402
from mixed_precision_optimizer_bf16_gb300.optimizer import BF16Optimizer, alloc_flat  # noqa: E402
from harness import GpuShard, check_norms, compare, ogroups, oracle_dense, oracle_sampled, sample_indices  # noqa: E402

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")


@pytest.fixture(autouse=True)
def _cleanup():
    yield
    gc.collect()
    if torch.cuda.is_available():
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def dense_parity(wl, defer=False, grad_scale=1.0, grad_per_tensor=False):
    sh = GpuShard(wl, grad_scale=grad_scale, defer=defer, grad_per_tensor=grad_per_tensor)
    sh.run(wl.steps)
    got = sh.states()
    norms = list(sh.norms)
    last_deferred = sh.defer
    sh.close()
    ref, scales = oracle_dense(wl, wl.steps, grad_scale)
    check_norms(norms, ref["sumsq"])
    return compare(got, ref, scales, wl, grad_scale, check_acc=not last_deferred)


def sampled_parity(wl, defer=False, k=1 << 15, extra=()):
    sh = GpuShard(wl, defer=defer)
    sh.run(wl.steps)
    idx = sample_indices(wl, k)
    if len(extra):
        idx = np.unique(np.concatenate([idx, np.asarray(extra, dtype=np.int64)]))
    got = sh.states(idx)
    norms = list(sh.norms)
    sh.close()
    del sh
    ref, scales = oracle_sampled(wl, wl.steps, idx)
    err = check_norms(norms, ref["sumsq"])
    st = compare(got, ref, scales, wl, check_acc=not defer)
    st["norm_rel_err"] = err
    return st


# ---------------------------------------------------------------- generators

@needs_cuda
def test_device_generator_matches_host():
    for wl in (workloads.workload(5), workloads.workload(2)):
        n = 1 << 20
        first = wl.n - n if wl.id == 2 else 12345
        d = torch.empty(n, dtype=torch.int16, device="cuda")
        sgpu.fill_grad(wl, 1, 1, d, first)
        h = synth.fill_grad(wl, 1, 1, np.empty(n, np.uint16), first)
        assert np.array_equal(d.cpu().numpy().view(np.uint16), h)
        f = torch.empty(n, dtype=torch.float32, device="cuda")
        sgpu.fill_master(wl, f, first)
        hm = synth.fill_master(wl, np.empty(n, np.float32), first)
        assert np.array_equal(f.cpu().numpy().view(np.uint32), hm.view(np.uint32))


# ------------------------------------------------------------- dense parity

@needs_cuda
@pytest.mark.parametrize("step", ["auto", "pipe"])
@pytest.mark.parametrize("defer", [False, True])
def test_tiny_workload_dense(defer, step, monkeypatch):
    """The 1M-element shard, 3 steps; "pipe": the fused step forced through the
    bulk-copy pipeline (a shard this small takes vector loads by default)."""
    if step == "pipe":
        monkeypatch.setenv("BF16OPT_PIPE", "1")
    st = dense_parity(workloads.workload(1), defer=defer)
    print("tiny", defer, step, st)


@needs_cuda
@pytest.mark.parametrize("defer", [False, True])
def test_clip_edge_workload_dense(defer):
    """2^27+13 elements, every buffer 2 elements past a 256-B boundary, clip ~1/163,
    1 % exact-zero gradients, masters log-uniform over 1e-8..1e3, 5 steps."""
    wl = workloads.workload(5)
    st = dense_parity(wl, defer=defer)
    print("clip edge", defer, st)


SMALL = [
    # (sizes, misalign, gas, steps, sigma)
    ([1], 0, 1, 2, 1e-3),
    ([2], 1, 2, 2, 0.5),
    ([3, 5], 3, 3, 2, 1e-3),
    ([7, 8, 9], 2, 2, 3, 0.2),
    ([31, 1000, 4096], 5, 2, 2, 1e-3),
    ([16383, 1, 16384, 16385], 7, 3, 2, 0.05),
    ([50001, 3], 6, 1, 3, 1e-2),
    ([65536 * 3 + 17], 4, 2, 2, 1e-3),
    ([4, 4, 4, 4], 0, 2, 2, 0.3),
]


@needs_cuda
@pytest.mark.parametrize("step", ["auto", "pipe"])
@pytest.mark.parametrize("case", range(len(SMALL)))
@pytest.mark.parametrize("mode", ["flat", "list"])
@pytest.mark.parametrize("defer", [False, True])
def test_small_ragged_variants(case, mode, defer, step, monkeypatch):
    if step == "pipe":
        monkeypatch.setenv("BF16OPT_PIPE", "1")
    sizes, mis, gas, steps, sigma = SMALL[case]
    decay = [(i % 3) != 1 for i in range(len(sizes))]
    wl = workloads.custom(100 + case, sizes, decay=decay, gas=gas, steps=steps, grad_sigma=sigma, misalign=mis,
                          mode=mode)
    dense_parity(wl, defer=defer)


@needs_cuda
@pytest.mark.parametrize("pat", [[False, False, True], [False, True, True], [True, True, True, True],
                                 [False, False, False], [True, False, True]])
def test_list_pipeline_with_own_gradient_buffers(pat, monkeypatch):
    """LIST tensors of ragged sizes whose gradients have buffers of their own,
    offset like their state (so the bulk-copy pipeline applies whatever the
    sizes), the pipeline forced: the later accumulates and the step fold the
    gradients -- the deferred ones too -- through bulk copies, with scalar
    heads and tails on every tensor, and equal the oracle over two steps."""
    monkeypatch.setenv("BF16OPT_PIPE", "1")
    monkeypatch.setenv("BF16OPT_SCHEDULE", "claim")
    wl = workloads.custom(275, [20_000, 5, 16_385, 1200, 7, 65_539], decay=[True, False, True, False, True, True],
                          gas=len(pat), steps=2, grad_sigma=0.05, misalign=3, mode="list")
    dense_parity(wl, defer=pat, grad_per_tensor=True)


@needs_cuda
@pytest.mark.parametrize("sched", ["auto", "claim", "pipe"])
def test_list_more_tensors_than_one_launch(sched, monkeypatch):
    """1100 tensors (> 1024 gradient pointers per launch): two launches per pass
    (three with two pointers per tensor) -- with claiming forced on, the
    launches of one pass share the chunk counter one after another; "pipe"
    also forces the fused step through the bulk-copy pipeline, whose launches
    share the counter the same way."""
    if sched in ("claim", "pipe"):
        monkeypatch.setenv("BF16OPT_SCHEDULE", "claim")
    if sched == "pipe":
        monkeypatch.setenv("BF16OPT_PIPE", "1")
    rng = np.random.default_rng(5)
    sizes = rng.integers(1, 700, 1100).tolist()
    wl = workloads.custom(150, sizes, decay=[i % 2 == 0 for i in range(1100)], gas=2, steps=2,
                          grad_sigma=0.05, misalign=3, mode="list")
    dense_parity(wl)
    dense_parity(wl, defer=True)
    dense_parity(wl, defer=[True, True])      # two pointers per tensor: 512 tensors per launch


@needs_cuda
def test_grad_scale():
    wl = workloads.custom(160, [70000, 333], decay=[True, False], gas=3, steps=2, grad_sigma=0.3)
    dense_parity(wl, grad_scale=0.25)
    dense_parity(wl, defer=True, grad_scale=0.25)


# ----------------------------------------------------------- full-size sampled

# (The full-size shards are compared on every element in
# test_full_size_dense_gpu.py.)


@needs_cuda
def test_flat_range_beyond_2_32_elements():
    """One flat range of 2^32 + 4099 elements (~86 GB on the device): 64-bit
    element offsets in the chunk table and the kernels, sampled on both sides
    of 2^31 and 2^32 and at the ragged end."""
    n = (1 << 32) + 4099
    wl = workloads.custom(270, [n], gas=2, steps=1, grad_sigma=1e-4)
    edges = [(1 << 31) + d for d in range(-3, 4)] + [(1 << 32) + d for d in range(-5, 6)] + [n - 1, n - 2, n - 4099]
    st = sampled_parity(wl, defer=True, k=1 << 14, extra=edges)
    print("beyond 2^32", st)


# ------------------------------------------------------------ behaviour

@needs_cuda
def test_determinism_bitwise():
    wl = workloads.custom(170, [300_000, 5000, 77], decay=[True, False, True], gas=3, steps=2, grad_sigma=0.1,
                          misalign=1)
    outs = []
    for _ in range(2):
        sh = GpuShard(wl, defer=True)
        sh.run(wl.steps)
        outs.append((sh.states(), list(sh.norms)))
        sh.close()
    (a, na), (b, nb) = outs
    assert na == nb
    for k in ("p", "m", "v", "p_bf16"):
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8))


def _raw_flat(n, groups=None):
    wl = workloads.custom(180, [max(n, 1)])
    flat = alloc_flat(n, "cuda")
    for k in flat:
        flat[k].zero_()
    desc = C.flat_desc(n, *(flat[k].data_ptr() if n else 0 for k in
                            ("master", "exp_avg", "exp_avg_sq", "grad_accum", "param_bf16")),
                       groups or wl.groups)
    rc, h = C.bf16opt_create(desc)
    assert rc == 0, C.bf16opt_last_error(None)
    return flat, h


@needs_cuda
def test_sequence_errors():
    flat, h = _raw_flat(1000)
    g = torch.zeros(1000, dtype=torch.int16, device="cuda")
    assert C.bf16opt_step(h) == C.BF16OPT_ERR_SEQUENCE
    assert C.bf16opt_grad_norm(h)[0] == C.BF16OPT_ERR_SEQUENCE
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, 0) == C.BF16OPT_ERR_SEQUENCE
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, C.BF16OPT_DEFER) == C.BF16OPT_ERR_SEQUENCE
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, 8) == C.BF16OPT_ERR_INVALID_ARG   # unknown flag
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, C.BF16OPT_FIRST) == 0
    assert C.bf16opt_step(h) == C.BF16OPT_ERR_SEQUENCE
    assert C.bf16opt_grad_norm(h, 0, True)[0] == C.BF16OPT_ERR_SEQUENCE        # no LAST micro-batch yet
    assert C.bf16opt_grad_norm_local(h)[0] == C.BF16OPT_ERR_SEQUENCE
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, C.BF16OPT_LAST) == 0
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, C.BF16OPT_LAST) == C.BF16OPT_ERR_SEQUENCE
    rc, nrm = C.bf16opt_grad_norm(h, 0, True)
    assert rc == 0 and nrm == 0.0
    assert C.bf16opt_step(h) == 0
    assert C.bf16opt_step(h) == C.BF16OPT_ERR_SEQUENCE
    assert C.bf16opt_get_step(h) == (0, 1)
    assert C.bf16opt_accumulate(h, g.data_ptr() + 1, None, C.BF16OPT_FIRST) == C.BF16OPT_ERR_ALIGNMENT
    assert "sequence" in C.bf16opt_error_string(C.BF16OPT_ERR_SEQUENCE)
    C.bf16opt_destroy(h)


@needs_cuda
@pytest.mark.parametrize("bad", [float("inf"), float("nan")])
def test_nonfinite_gradient_warns(bad):
    flat, h = _raw_flat(5000)
    g = torch.zeros(5000, dtype=torch.float32, device="cuda")
    g[1234] = bad
    gb = g.to(torch.bfloat16).view(torch.int16)
    assert C.bf16opt_accumulate(h, gb.data_ptr(), None, C.BF16OPT_FIRST | C.BF16OPT_LAST) == 0
    rc, nrm = C.bf16opt_grad_norm(h, 0, True)
    assert rc == C.BF16OPT_WARN_NONFINITE
    assert math.isinf(nrm) and nrm > 0 if math.isinf(bad) else math.isnan(nrm)   # sqrt of the FP64 sum
    assert C.bf16opt_step(h) == 0  # the library does not skip; the caller decides
    torch.cuda.synchronize()
    C.bf16opt_destroy(h)


@needs_cuda
def test_empty_shard():
    flat, h = _raw_flat(0)
    assert C.bf16opt_accumulate(h, 0, None, C.BF16OPT_FIRST | C.BF16OPT_LAST) == 0
    assert C.bf16opt_grad_norm(h, 0, True) == (0, 0.0)
    assert C.bf16opt_step(h) == 0
    assert C.bf16opt_get_step(h) == (0, 1)
    assert C.bf16opt_step_path(h) == (0, C.BF16OPT_PATH_NONE)   # nothing to launch
    C.bf16opt_destroy(h)


@needs_cuda
def test_lr_override_and_resume():
    """lr_override replaces the groups' lr for one step; a new handle over the
    same buffers with set_step(2) continues exactly like an uninterrupted run."""
    wl = workloads.custom(190, [20000, 1000], decay=[True, False], gas=2, steps=3, grad_sigma=0.2)
    # uninterrupted 3 steps with lr x0.5 on the last step
    sh = GpuShard(wl)
    sh.run_step(0)
    sh.run_step(1)
    for k in range(wl.gas):
        sgpu.fill_grad(wl, 2, k, sh.gbuf)
        sh.opt.accumulate(sh.gbuf, first=k == 0, last=k == wl.gas - 1)
    sh.opt.grad_norm()
    sh.opt.step(lr=[3e-5, 3e-5])
    a = sh.states()
    sh.close()
    # interrupted: 2 steps, new handle, set_step(2), last step
    sh2 = GpuShard(wl)
    sh2.run_step(0)
    sh2.run_step(1)
    sh2.opt.close()
    sh2.opt = BF16Optimizer(wl.groups, flat=sh2.flat, ranges=wl.ranges(), max_grad_norm=wl.max_norm)
    sh2.opt.t = 2
    for k in range(wl.gas):
        sgpu.fill_grad(wl, 2, k, sh2.gbuf)
        sh2.opt.accumulate(sh2.gbuf, first=k == 0, last=k == wl.gas - 1)
    sh2.opt.grad_norm()
    sh2.opt.step(lr=[3e-5, 3e-5])
    b = sh2.states()
    assert sh2.opt.t == 3
    sh2.close()
    for k in ("p", "m", "v", "p_bf16"):
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8))
    # and the oracle with lr 3e-5 on step 3
    import harness
    G = ogroups(wl)
    n = wl.n
    gof = wl.group_of(np.arange(n))
    p = synth.fill_master(wl, np.empty(n, np.float32))
    sc = {"M": np.zeros(n), "A": np.abs(p.astype(np.float64))}
    gfn = lambda s, k: synth.fill_grad(wl, s, k, np.empty(n, np.uint16))
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    lr3 = float(np.float32(3e-5))
    for s in range(3):
        Gs = G if s < 2 else [oracle.group(lr3, g.beta1, g.beta2, g.eps, g.weight_decay) for g in G]
        r = oracle.run_dense(p, gfn, wl.ranges(), Gs, 1, wl.gas, wl.max_norm, t0=s, m=m, v=v)
        p, m, v = r["p"], r["m"], r["v"]
        if s == 2:
            wl.groups = [dict(g, lr=3e-5) for g in wl.groups]
        harness._update_scales(sc, wl, gof, r["acc"], r["clip"][0], m, v, s + 1, 1.0)
    compare(a, r, sc, wl)


@needs_cuda
@pytest.mark.parametrize("pipe", ["0", "1"])
def test_step_kernel_follows_the_switch(pipe, monkeypatch):
    """BF16OPT_PIPE=1 runs the fused step as the bulk-copy pipeline
    kernel, =0 as the vector-load kernel -- so the tests that force either one
    exercise the kernel they name."""
    monkeypatch.setenv("BF16OPT_PIPE", pipe)
    wl = workloads.custom(196, [20_001, 77], decay=[True, False], gas=2, steps=1, grad_sigma=0.1, misalign=3)
    sh = GpuShard(wl, defer=True)
    assert C.bf16opt_step_path(sh.opt.h) == (0, C.BF16OPT_PATH_NONE)
    sh.run(1)
    want = C.BF16OPT_PATH_PIPELINE if pipe == "1" else C.BF16OPT_PATH_VECTOR
    assert C.bf16opt_step_path(sh.opt.h) == (0, want)
    sh.close()


@needs_cuda
def test_pipe_needs_bf16_offsets_alike():
    """Gradients 4 elements (8 bytes) off the parameters' offset modulo 16 bytes:
    vector loads still apply (same offset modulo 8 bytes) but no element puts
    every bf16 stream on a 16-byte boundary, so the step takes the vector-load
    kernel even when the pipeline is asked for -- and equals the oracle."""
    import os
    wl = workloads.custom(197, [10_007, 64], decay=[True, False], gas=2, steps=2, grad_sigma=0.1)
    n = wl.n
    os.environ["BF16OPT_PIPE"] = "1"
    try:
        flat = {k: torch.zeros(n, dtype=dt, device="cuda") for k, dt in
                (("master", torch.float32), ("exp_avg", torch.float32), ("exp_avg_sq", torch.float32),
                 ("grad_accum", torch.float32), ("param_bf16", torch.int16))}
        sgpu.fill_master(wl, flat["master"])
        opt = BF16Optimizer(wl.groups, flat=flat, ranges=wl.ranges(), max_grad_norm=wl.max_norm)
    finally:
        os.environ.pop("BF16OPT_PIPE", None)
    gb = torch.empty(n + 64, dtype=torch.int16, device="cuda")[4:4 + n]
    norms = []

    def one(s):
        for k in range(wl.gas):
            sgpu.fill_grad(wl, s, k, gb)
            opt.accumulate(gb, first=k == 0, last=k == wl.gas - 1, defer=k == wl.gas - 1)
        norms.append(opt.grad_norm(sync=True))
        opt.step()

    one(0)
    assert C.bf16opt_step_path(opt.h) == (0, C.BF16OPT_PATH_VECTOR)
    one(1)
    got = dict(p=flat["master"].cpu().numpy(), m=flat["exp_avg"].cpu().numpy(), v=flat["exp_avg_sq"].cpu().numpy(),
               acc=flat["grad_accum"].cpu().numpy(), p_bf16=flat["param_bf16"].cpu().numpy().view(np.uint16))
    opt.close()
    ref, scales = oracle_dense(wl, wl.steps)
    check_norms(norms, ref["sumsq"])
    compare(got, ref, scales, wl, check_acc=False)


@needs_cuda
def test_inconsistent_alignment_falls_back_correctly():
    """Buffers with different offsets modulo 16 B take the element-wise path."""
    wl = workloads.custom(195, [10007], gas=2, steps=2, grad_sigma=0.1)
    n = wl.n
    bufs = {}
    for i, (k, dt) in enumerate((("master", torch.float32), ("exp_avg", torch.float32), ("exp_avg_sq", torch.float32),
                                 ("grad_accum", torch.float32), ("param_bf16", torch.int16))):
        base = torch.zeros(n + 64, dtype=dt, device="cuda")
        bufs[k] = base[i % 4:i % 4 + n]
    sgpu.fill_master(wl, bufs["master"])
    opt = BF16Optimizer(wl.groups, flat=bufs, ranges=wl.ranges(), max_grad_norm=wl.max_norm)
    gb = torch.empty(n + 64, dtype=torch.int16, device="cuda")[3:3 + n]
    norms = []
    for s in range(wl.steps):
        for k in range(wl.gas):
            sgpu.fill_grad(wl, s, k, gb)
            opt.accumulate(gb, first=k == 0, last=k == wl.gas - 1)
        norms.append(opt.grad_norm(sync=True))
        opt.step()
    got = dict(p=bufs["master"].cpu().numpy(), m=bufs["exp_avg"].cpu().numpy(), v=bufs["exp_avg_sq"].cpu().numpy(),
               acc=bufs["grad_accum"].cpu().numpy(), p_bf16=bufs["param_bf16"].cpu().numpy().view(np.uint16))
    opt.close()
    ref, scales = oracle_dense(wl, wl.steps)
    check_norms(norms, ref["sumsq"])
    compare(got, ref, scales, wl)


# ------------------------------------------------------------ guard bands

PAD = 256  # elements of canary on each side of every buffer


def _guarded(n, dtype, mis):
    """A buffer of n elements `mis` elements into an allocation whose 256-element
    pads on both sides hold a NaN canary pattern."""
    base = torch.empty(n + 2 * PAD + 8, dtype=dtype, device="cuda")
    if dtype == torch.float32:
        base.view(torch.int32).fill_(0x7FC00D0D)
    else:
        base.fill_(0x7FCD)
    return base, base[PAD + mis:PAD + mis + n]


def _pads_intact(base, n, mis):
    a = base.view(torch.int32 if base.dtype == torch.float32 else torch.int16).cpu().numpy()
    want = 0x7FC00D0D if base.dtype == torch.float32 else 0x7FCD
    head, tail = a[:PAD + mis], a[PAD + mis + n:]
    return bool((head == want).all() and (tail == want).all())


@needs_cuda
@pytest.mark.parametrize("mode", ["flat", "list"])
def test_guard_bands_untouched(mode):
    """No kernel writes outside its buffers and the gradients are only read."""
    sizes = [16385, 3, 40001] if mode == "list" else [56389]
    wl = workloads.custom(220, sizes, decay=[True, False, True][:len(sizes)], gas=3, steps=2, grad_sigma=0.1,
                          misalign=3, mode=mode)
    keys = ("master", "exp_avg", "exp_avg_sq", "grad_accum", "param_bf16")
    bases, views = [], []
    tensors = []
    for t in wl.tensors:
        d = {}
        for k in keys:
            b, v = _guarded(t.numel, torch.int16 if k == "param_bf16" else torch.float32, wl.misalign)
            v.zero_()
            bases.append((b, t.numel))
            d[k] = v
        sgpu.fill_master(workloads.custom(220, [t.numel]), d["master"])
        d["group"] = 0
        tensors.append(d)
    gb, g = _guarded(wl.n, torch.int16, wl.misalign)
    if mode == "flat":
        opt = BF16Optimizer(wl.groups, flat=tensors[0], ranges=wl.ranges(), max_grad_norm=1.0)
        garg = g
    else:
        opt = BF16Optimizer(wl.groups, tensors=tensors, max_grad_norm=1.0)
        garg = [g[o:o + t.numel] for t, o in zip(wl.tensors, wl.offsets)]
    for s in range(wl.steps):
        for k in range(wl.gas):
            sgpu.fill_grad(wl, s, k, g)
            before = g.clone()
            opt.accumulate(garg, first=k == 0, last=k == wl.gas - 1, defer=(s == 1 and k == wl.gas - 1))
        opt.grad_norm()
        opt.step()
        torch.cuda.synchronize()
        assert torch.equal(g, before)                  # gradients are read-only
    opt.close()
    for b, n in bases:
        assert _pads_intact(b, n, wl.misalign)
    assert _pads_intact(gb, wl.n, wl.misalign)


# ------------------------------------------------------- multi-rank norm hooks

@needs_cuda
def test_two_partitions_share_the_global_norm():
    """Two handles over the two halves of one shard stand for two ZeRO ranks
    (their calls are sequenced on the host; no kernel waits on another).  Each
    reports its local sum of squares, the sum in rank order is handed back to
    both, and the two halves then step exactly like the whole shard would."""
    wl = workloads.custom(230, [70_000, 333, 50_001], decay=[True, False, True], gas=3, steps=2, grad_sigma=0.2)
    n, half = wl.n, 60_000
    flat = alloc_flat(wl.n, "cuda")
    sgpu.fill_master(wl, flat["master"])
    for k in ("exp_avg", "exp_avg_sq", "grad_accum", "param_bf16"):
        flat[k].zero_()
    parts = [{k: v[:half] for k, v in flat.items()}, {k: v[half:] for k, v in flat.items()}]

    def local_ranges(lo, hi):
        return [(max(b, lo) - lo, min(e, hi) - lo, g) for b, e, g in wl.ranges() if max(b, lo) < min(e, hi)]

    opts = [BF16Optimizer(wl.groups, flat=parts[0], ranges=local_ranges(0, half)),
            BF16Optimizer(wl.groups, flat=parts[1], ranges=local_ranges(half, n))]
    g = torch.empty(n, dtype=torch.int16, device="cuda")
    norms = []
    for s in range(wl.steps):
        for k in range(wl.gas):
            sgpu.fill_grad(wl, s, k, g)
            opts[0].accumulate(g[:half], first=k == 0, last=k == wl.gas - 1)
            opts[1].accumulate(g[half:], first=k == 0, last=k == wl.gas - 1)
        locs = []
        for o in opts:
            rc, loc = C.bf16opt_grad_norm_local(o.h, torch.cuda.current_stream().cuda_stream)
            assert rc == 0
            locs.append(loc)
        got_norms = []
        for r, o in enumerate(opts):
            if locs[0] != locs[1]:   # values gathered out of rank order are refused
                assert C.bf16opt_set_rank_sumsqs(o.h, locs[::-1], r)[0] == C.BF16OPT_ERR_INVALID_ARG
            rc, nrm = C.bf16opt_set_rank_sumsqs(o.h, locs, r, torch.cuda.current_stream().cuda_stream)
            assert rc == 0, C.bf16opt_last_error(o.h)
            got_norms.append(nrm)
            o.step()
        assert got_norms[0] == got_norms[1] == math.sqrt(locs[0] + locs[1])
        norms.append(got_norms[0])
    torch.cuda.synchronize()
    got = dict(p=flat["master"].cpu().numpy(), m=flat["exp_avg"].cpu().numpy(),
               v=flat["exp_avg_sq"].cpu().numpy(), acc=flat["grad_accum"].cpu().numpy(),
               p_bf16=flat["param_bf16"].cpu().numpy().view(np.uint16))
    for o in opts:
        assert C.bf16opt_set_global_sumsq(o.h, 1.0) == C.BF16OPT_ERR_SEQUENCE
        o.close()
    ref, scales = oracle_dense(wl, wl.steps)
    check_norms(norms, ref["sumsq"])
    compare(got, ref, scales, wl)


# ------------------------------------------------- deferred micro-batches

DEFER_PATTERNS = [
    [True, True, True, True],                  # nothing stored: norm and step fold all four
    [True, False, True, True],                 # pairs: one stored pass, then the last two deferred
    [True, False, False, False],
    [False, True, True, False],
    [True, True, False],
    [True] * 5,                                # five pending (8-wide kernels, runtime count 5)
    [True] * 8,                                # the maximum
    [False, True, False, True, False, True, True],
    [True] * 8 + [False],                      # 8 pending, then a stored pass: pre-fold, then this one
    [True] * 8 + [False, True],                # ... and a deferred last micro-batch after it
    [False] + [True] * 8 + [False, False],     # the pre-fold onto a stored accumulator
    [True] * 7 + [False] + [True] * 7 + [False] + [True],   # runs of 8 folded by their 8th (GAS 17)
]


@needs_cuda
@pytest.mark.parametrize("step", ["auto", "pipe"])
@pytest.mark.parametrize("pat", range(len(DEFER_PATTERNS)))
@pytest.mark.parametrize("mode", ["flat", "list"])
def test_deferred_patterns(pat, mode, step, monkeypatch):
    """Deferring any micro-batches folds the same FP32 adds in the same order
    (with "pipe", in the bulk-copy step too: up to 8 gradient slots per stage)."""
    if step == "pipe":
        monkeypatch.setenv("BF16OPT_PIPE", "1")
    pattern = DEFER_PATTERNS[pat]
    sizes = [50_001, 3, 16_384, 777] if mode == "flat" else [20_000, 5, 16_385, 1200]
    wl = workloads.custom(240 + pat, sizes, decay=[True, False, True, False], gas=len(pattern), steps=2,
                          grad_sigma=0.05, misalign=pat % 4, mode=mode)
    st = dense_parity(wl, defer=pattern)
    print(mode, pattern, st)


@needs_cuda
def test_too_many_deferred():
    flat, h = _raw_flat(4096)
    g = torch.zeros(4096, dtype=torch.int16, device="cuda")
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, C.BF16OPT_FIRST | C.BF16OPT_DEFER) == 0
    for _ in range(C.BF16OPT_MAX_DEFERRED - 1):
        assert C.bf16opt_accumulate(h, g.data_ptr(), None, C.BF16OPT_DEFER) == 0
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, C.BF16OPT_DEFER) == C.BF16OPT_ERR_INVALID_ARG
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, C.BF16OPT_LAST) == 0   # a stored pass folds all nine
    assert C.bf16opt_grad_norm(h, 0, True) == (0, 0.0)
    assert C.bf16opt_step(h) == 0
    torch.cuda.synchronize()
    C.bf16opt_destroy(h)


@needs_cuda
def test_results_do_not_depend_on_the_grid(monkeypatch):
    """The norm's partials belong to chunks, not CTAs, and the step is
    element-wise: one CTA per launch gives the same bits as the full grid,
    and so does any grid whose CTAs claim their chunks from the counter (in
    whatever order the claims land) instead of taking a fixed stride."""
    wl = workloads.custom(250, [300_001, 4097, 77], decay=[True, False, True], gas=3, steps=2, grad_sigma=0.1,
                          misalign=1)
    outs = []
    for cap, sched, pipe in ((None, "static", "0"), ("1", "static", "0"), ("7", "static", "0"), (None, "claim", "0"),
                             ("1", "claim", "0"), ("7", "claim", "0"), (None, "static", "1"), ("1", "static", "1"),
                             ("7", "claim", "1"), (None, "claim", "1")):
        monkeypatch.setenv("BF16OPT_SCHEDULE", sched)
        monkeypatch.setenv("BF16OPT_PIPE", pipe)
        if cap is None:
            monkeypatch.delenv("BF16OPT_MAX_GRID", raising=False)
        else:
            monkeypatch.setenv("BF16OPT_MAX_GRID", cap)
        sh = GpuShard(wl, defer=[True, False, True])
        sh.run(wl.steps)
        outs.append((sh.states(), list(sh.norms)))
        sh.close()
    for st, nr in outs[1:]:
        assert nr == outs[0][1]
        for k in ("p", "m", "v", "p_bf16"):
            assert np.array_equal(st[k].view(np.uint8), outs[0][0][k].view(np.uint8))


# ------------------------------------------------------------ CUDA graphs

@needs_cuda
@pytest.mark.parametrize("sched", ["auto", "claim", "pipe"])
@pytest.mark.parametrize("mode", ["flat", "list"])
def test_cuda_graph_replay_matches_eager(mode, sched, monkeypatch):
    """One step captured into a CUDA graph and replayed for the later steps
    (fresh gradients written into the same buffers before each replay) gives
    the same bits as calling the API eagerly: the step counter and the
    per-step scalars live on the device.  With chunk claiming forced on, the
    replays also show that the claim counter is back at zero after every pass
    (it resets itself; no memset node sits in the graph)."""
    if sched in ("claim", "pipe"):
        monkeypatch.setenv("BF16OPT_SCHEDULE", "claim")
    if sched == "pipe":
        monkeypatch.setenv("BF16OPT_PIPE", "1")
    wl = workloads.custom(260, [40_000, 3, 16_385, 999], decay=[True, False, True, False], gas=3, steps=4,
                          grad_sigma=0.1, misalign=2, mode=mode)
    eager = GpuShard(wl, defer=[False, True, True])
    eager.opt.set_lr_schedule(2, 4, 0.5)
    eager.run(wl.steps)
    want = eager.states()
    eager.close()

    sh = GpuShard(wl, defer=[False, True, True])
    sh.opt.set_lr_schedule(2, 4, 0.5)
    sh.run_step(0)                                # eager warm-up: loads every kernel
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for k in range(wl.gas):
            sh.opt.accumulate(sh.grads_arg(sh.gbufs[k % len(sh.gbufs)]), first=k == 0, last=k == wl.gas - 1,
                              defer=sh.pattern[k])
        sh.opt.grad_norm()
        sh.opt.step()
    for s in range(1, wl.steps):
        for k in range(wl.gas):
            sgpu.fill_grad(wl, s, k, sh.gbufs[k % len(sh.gbufs)])
        graph.replay()
    torch.cuda.synchronize()
    got = sh.states()
    assert sh.opt.t == wl.steps
    sh.close()
    for k in ("p", "m", "v", "p_bf16"):
        assert np.array_equal(got[k].view(np.uint8), want[k].view(np.uint8)), k


@needs_cuda
def test_pinned_host_buffer_round_trip():
    from host_buffers import PinnedHostBuffer
    hb = PinnedHostBuffer(5_000_003, torch.int16)
    assert hb.tensor.is_pinned() and hb.tensor.numel() == 5_000_003
    d = torch.randint(-30000, 30000, (5_000_003,), dtype=torch.int16, device="cuda")
    hb.tensor.copy_(d)
    e = torch.empty_like(d)
    e.copy_(hb.tensor, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(d, e)
    hb.close()


@needs_cuda
@pytest.mark.parametrize("mode", ["flat", "list"])
def test_checkpoint_dump_free_restore(mode):
    """Checkpoint/resume: the state is the caller's buffers plus the step
    counter.  Two steps, dump master/m/v/bf16 to host memory, free the handle
    and every buffer, restore into freshly allocated buffers, set the step
    counter, one more step == three uninterrupted steps, bit for bit."""
    wl = workloads.custom(280, [30_001, 7, 16_385], decay=[True, False, True], gas=3, steps=3, grad_sigma=0.2,
                          misalign=1, mode=mode)
    ref = GpuShard(wl, defer=True)
    ref.run(3)
    want = ref.states()
    ref.close()
    del ref

    sh = GpuShard(wl, defer=True)
    sh.run_step(0)
    sh.run_step(1)
    torch.cuda.synchronize()
    saved = {k: v.copy() for k, v in sh.states().items()}
    t_saved = sh.opt.t
    sh.close()
    del sh
    gc.collect()
    torch.cuda.empty_cache()

    # fresh buffers with the same offset modulo 16 bytes: the norm's per-chunk
    # partials follow the thread->element map, which that offset fixes
    wl2 = workloads.custom(280, [30_001, 7, 16_385], decay=[True, False, True], gas=3, steps=3, grad_sigma=0.2,
                           misalign=1, mode=mode)
    sh2 = GpuShard(wl2, defer=True)
    names = dict(p="master", m="exp_avg", v="exp_avg_sq", p_bf16="param_bf16")
    for key, name in names.items():
        host = torch.from_numpy(saved[key].view(np.int16) if key == "p_bf16" else saved[key])
        if wl2.mode == "flat":
            sh2.flat[name].copy_(host)
        else:
            for d, t, off in zip(sh2.tensors, wl2.tensors, wl2.offsets):
                d[name].copy_(host[off:off + t.numel])
    sh2.opt.t = t_saved
    sh2.run_step(2)
    got = sh2.states()
    assert sh2.opt.t == 3
    sh2.close()
    for k in ("p", "m", "v", "p_bf16"):
        assert np.array_equal(got[k].view(np.uint8), want[k].view(np.uint8)), k


@needs_cuda
@pytest.mark.parametrize("use_graph", [False, True])
def test_skip_nonfinite_step(use_graph):
    """With skipping enabled a step whose norm is Inf leaves every state buffer
    and the step counter untouched (decided on the device, so it also works in
    a replayed graph); the next clean step continues exactly like a run that
    never saw the bad step."""
    import harness
    wl = workloads.custom(290, [20_000, 333], decay=[True, False], gas=2, steps=2, grad_sigma=0.1, misalign=1)
    ref = GpuShard(wl)
    ref.run(2)                                   # steps 0 and 1, no bad step
    want = ref.states()
    ref.close()

    sh = GpuShard(wl)
    sh.opt.set_skip_nonfinite(True)
    sh.run_step(0)
    torch.cuda.synchronize()
    before = sh.states()
    bufs = [harness._alloc(wl.n, torch.int16, wl.misalign) for _ in range(wl.gas)]   # one per micro-batch

    def enqueue():
        for k in range(wl.gas):
            sh.opt.accumulate(bufs[k], first=k == 0, last=k == wl.gas - 1)
        sh.opt.grad_norm()
        sh.opt.step()

    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            enqueue()

    def step_with(step_index, poison):
        for k in range(wl.gas):
            sgpu.fill_grad(wl, step_index, k, bufs[k])
        if poison:
            bufs[1][123] = 0x7F80                    # bf16 +Inf in micro-batch 1
        if graph is None:
            enqueue()
        else:
            graph.replay()
        torch.cuda.synchronize()

    step_with(1, poison=True)
    skipped = sh.states()
    assert sh.opt.t == 1
    for k in ("p", "m", "v", "p_bf16"):
        assert np.array_equal(skipped[k].view(np.uint8), before[k].view(np.uint8)), k
    step_with(1, poison=False)
    assert sh.opt.t == 2
    got = sh.states()
    sh.close()
    for k in ("p", "m", "v", "p_bf16"):
        assert np.array_equal(got[k].view(np.uint8), want[k].view(np.uint8)), k


@needs_cuda
def test_step_counter_calls_wait_for_steps_on_side_streams():
    """get_step, set_step and the set_* calls are ordered after a step still in
    flight on a non-blocking stream: a sleep kernel (about 20 ms) holds the
    stream, so a plain copy on the legacy stream would read or write the
    counter before the step's own increment."""
    wl = workloads.custom(291, [50_000, 77], decay=[True, False], gas=1, steps=3, grad_sigma=0.1)
    sh = GpuShard(wl)
    side = torch.cuda.Stream()

    def step_on_side(step_index):
        sgpu.fill_grad(wl, step_index, 0, sh.gbuf)
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            torch.cuda._sleep(40_000_000)
            sh.opt.accumulate(sh.grads_arg(), first=True, last=True, stream=side)
            sh.opt.grad_norm(stream=side)
            sh.opt.step(stream=side)

    step_on_side(0)
    assert sh.opt.t == 1                 # read waits for the step behind the sleep
    step_on_side(1)
    sh.opt.t = 10                        # write is ordered after that step (t = 2 there)
    torch.cuda.synchronize()
    assert sh.opt.t == 10
    step_on_side(2)
    sh.opt.set_skip_nonfinite(False)     # waits too; the step completes first
    assert sh.opt.t == 11
    sh.close()


# Gradient elements whose squares exceed FP32's range (bf16 has FP32's exponent
# range, so these are ordinary bf16 values), placed in the head, vector body and
# ragged tail of several chunks and in both tensors.  The largest dominates the
# norm (about 2.5e30), so the clip coefficient and every stored moment stay
# normal FP32 numbers.
BIG_GRADS = {1: 1.5e19, 40_000: -3e25, 40_001: 2.5e30, 65_537: 1e20, 70_000: -7e19, 70_100: 4e22}


def _big_gradient_workload():
    wl = workloads.custom(292, [70_001, 333], decay=[True, False], gas=2, steps=1, grad_sigma=0.1, misalign=1)
    grads = [synth.fill_grad(wl, 0, k, np.empty(wl.n, np.uint16)) for k in range(wl.gas)]
    for i, x in BIG_GRADS.items():
        grads[i % 2][i] = int(np.float32(x).view(np.uint32)) >> 16     # bf16 by truncation
    return wl, grads


@needs_cuda
@pytest.mark.parametrize("variant", ["stored_last", "defer_last", "all_deferred"])
def test_gradients_whose_squares_overflow_fp32(variant):
    """The definition's sum of squares is FP64, where 2.5e30 squared is an
    ordinary number: the norm must be finite and equal the oracle's, the clip
    must bring the gradient to norm 1, and the step must match element by
    element -- on every pass that computes the norm's partials (stored LAST,
    deferred LAST, all deferred)."""
    import harness
    wl, grads = _big_gradient_workload()
    pattern = {"stored_last": [False, False], "defer_last": [False, True], "all_deferred": [True, True]}[variant]
    sh = GpuShard(wl, defer=pattern)
    for k in range(wl.gas):
        buf = sh.gbufs[k % len(sh.gbufs)]
        buf.copy_(torch.from_numpy(grads[k].view(np.int16)))
        sh.opt.accumulate(sh.grads_arg(buf), first=k == 0, last=k == wl.gas - 1, defer=pattern[k])
    norm = sh.opt.grad_norm(sync=True)
    sh.opt.step()
    torch.cuda.synchronize()
    got = sh.states()
    sh.close()

    p0 = synth.fill_master(wl, np.empty(wl.n, np.float32))
    ref = oracle.run_dense(p0.copy(), lambda s, k: grads[k], wl.ranges(), ogroups(wl), 1, wl.gas, wl.max_norm)
    S = ref["sumsq"][0]
    assert math.isfinite(S) and S > 6e60
    assert math.isfinite(norm) and abs(norm - math.sqrt(S)) <= harness.REL * math.sqrt(S)
    sc = {"M": np.zeros(wl.n), "A": np.abs(p0.astype(np.float64))}
    harness._update_scales(sc, wl, wl.group_of(np.arange(wl.n)), ref["acc"], ref["clip"][0], ref["m"], ref["v"],
                           1, 1.0)
    compare(got, ref, sc, wl, check_acc=variant == "stored_last")


@needs_cuda
@pytest.mark.parametrize("mode", ["flat", "list"])
def test_python_binding_rejects_mismatched_arguments(mode):
    """Gradients of the wrong dtype (FP32, FP16), size, layout or device, a
    gradient list of the wrong length, and a per-group lr list of the wrong
    length are refused in Python, before the library could read past a buffer;
    the handle's sequence is untouched and the next correct step matches the
    oracle."""
    wl = workloads.custom(293, [5000, 77], decay=[True, False], gas=1, steps=1, grad_sigma=0.1, mode=mode)
    sh = GpuShard(wl)
    k0 = wl.n if mode == "flat" else 5000           # the first (or only) gradient tensor
    bad = [torch.zeros(k0, dtype=torch.float32, device="cuda"),
           torch.zeros(k0, dtype=torch.float16, device="cuda"),
           torch.zeros(k0 + 1, dtype=torch.int16, device="cuda"),
           torch.zeros(2 * k0, dtype=torch.int16, device="cuda")[::2],
           torch.zeros(k0, dtype=torch.int16)]
    good_tail = torch.zeros(77, dtype=torch.int16, device="cuda")
    for b in bad:
        with pytest.raises(ValueError):
            sh.opt.accumulate(b if mode == "flat" else [b, good_tail], first=True, last=True)
    if mode == "list":
        with pytest.raises(ValueError, match="tensors"):
            sh.opt.accumulate(sh.grads_arg()[:1], first=True, last=True)
    sgpu.fill_grad(wl, 0, 0, sh.gbuf)
    sh.opt.accumulate(sh.grads_arg(), first=True, last=True)
    sh.opt.grad_norm(sync=True)
    with pytest.raises(ValueError, match="rates"):
        sh.opt.step(lr=[1e-4, 1e-4, 1e-4])
    sh.opt.step()
    torch.cuda.synchronize()
    got = sh.states()
    sh.close()
    ref, scales = oracle_dense(wl, 1)
    compare(got, ref, scales, wl)


def _random_case(seed):
    """A seeded random workload and micro-batch deferral pattern: GAS 1..12,
    1..5 tensors of 1..40,000 elements, FLAT or LIST, misaligned 0..7, and any
    defer pattern the library accepts (at most 8 deferred micro-batches pending
    at once; a stored micro-batch after 8 pending makes the library fold them
    first)."""
    rng = np.random.default_rng(7_000 + seed)
    gas = int(rng.integers(1, 13))
    pattern, pending = [], 0
    for _ in range(gas):
        d = bool(rng.integers(0, 2)) and pending < 8
        pattern.append(d)
        pending = pending + 1 if d else 0
    ntens = int(rng.integers(1, 6))
    sizes = [int(x) for x in rng.integers(1, 40_000, ntens)]
    wl = workloads.custom(400 + seed, sizes, decay=[bool(x) for x in rng.integers(0, 2, ntens)], gas=gas, steps=2,
                          grad_sigma=float(rng.choice([1e-3, 0.05, 0.5])), misalign=int(rng.integers(0, 8)),
                          mode="list" if seed % 2 else "flat")
    return wl, pattern, float(rng.choice([1.0, 0.5, 3.0]))


@needs_cuda
@pytest.mark.parametrize("seed", range(16))
def test_random_sequences_match_oracle(seed, monkeypatch):
    """Random shapes, layouts, GAS and deferral patterns: every one equals the
    oracle (norms, m, v, master, bf16) over two steps.  Half of the seeds
    force chunk claiming on (these shards are small enough to take the fixed
    stride by default), half force the fused step through the bulk-copy
    pipeline."""
    if seed % 4 in (1, 2):
        monkeypatch.setenv("BF16OPT_SCHEDULE", "claim")
    if seed % 4 in (2, 3):
        monkeypatch.setenv("BF16OPT_PIPE", "1")
    wl, pattern, gscale = _random_case(seed)
    dense_parity(wl, defer=pattern, grad_scale=gscale)


@needs_cuda
def test_destroyed_handle_is_rejected():
    """After bf16opt_destroy the handle value is refused by every call, and a
    second destroy is an error, not a double free."""
    flat, h = _raw_flat(1000)
    g = torch.zeros(1000, dtype=torch.int16, device="cuda")
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, C.BF16OPT_FIRST | C.BF16OPT_LAST) == 0
    assert C.bf16opt_destroy(h) == 0
    E = C.BF16OPT_ERR_INVALID_ARG
    assert C.bf16opt_grad_norm(h, 0, True)[0] == E
    assert C.bf16opt_step(h) == E
    assert C.bf16opt_accumulate(h, g.data_ptr(), None, C.BF16OPT_FIRST) == E
    assert C.bf16opt_get_step(h)[0] == E
    assert C.bf16opt_destroy(h) == E
    assert "not a live" in C.bf16opt_last_error(h)
    flat2, h2 = _raw_flat(1000)                  # a new handle works normally
    assert C.bf16opt_accumulate(h2, g.data_ptr(), None, C.BF16OPT_FIRST | C.BF16OPT_LAST) == 0
    assert C.bf16opt_destroy(h2) == 0


@needs_cuda
@pytest.mark.parametrize("mode", ["flat", "list"])
def test_state_dict_file_round_trip(tmp_path, mode):
    """Checkpoint through the Python API and a file: two steps with an LR
    schedule and skipping enabled, state_dict() saved with torch.save, every
    buffer freed, a fresh optimizer over new buffers (same offset modulo 128
    bytes) loads it and takes the third step -- equal, bit for bit, to three
    uninterrupted steps."""
    wl = workloads.custom(294, [30_001, 7, 16_385], decay=[True, False, True], gas=2, steps=3, grad_sigma=0.2,
                          misalign=3, mode=mode)

    def configure(opt):
        opt.set_lr_schedule(1, 10, 0.1)
        opt.set_skip_nonfinite(True)

    ref = GpuShard(wl, defer=True)
    configure(ref.opt)
    ref.run(3)
    want = ref.states()
    ref.close()
    del ref

    sh = GpuShard(wl, defer=True)
    configure(sh.opt)
    sh.run_step(0)
    sh.run_step(1)
    path = tmp_path / "opt.pt"
    torch.save(sh.opt.state_dict(), path)
    sh.close()
    del sh
    gc.collect()
    torch.cuda.empty_cache()

    sh2 = GpuShard(wl, defer=True)             # fresh buffers, fresh handle, default settings
    sd = torch.load(path, weights_only=True)      # plain tensors, numbers and lists
    sh2.opt.load_state_dict(sd)
    assert sh2.opt.t == 2
    sh2.run_step(2)
    got = sh2.states()
    sh2.close()
    for k in ("p", "m", "v", "p_bf16"):
        assert np.array_equal(got[k].view(np.uint8), want[k].view(np.uint8)), k


SWEEP_SIZES = [1, 2, 3, 4, 5, 7, 8, 31, 32, 33, 63, 64, 65, 2047, 2048, 2049, 4095, 4096, 4097]


@needs_cuda
@pytest.mark.parametrize("mode", ["flat", "list"])
def test_small_sizes_every_misalignment(mode):
    """Every buffer offset 0..7 elements for sizes around the quad, warp and
    128-byte boundaries (1 ... 4097 elements; LIST adds a second, 5-element
    tensor), GAS cycling 1, 2, 3 and the last micro-batch deferred on every
    other case, the fused step through vector loads and through the bulk-copy
    pipeline: 304 dense runs, each equal to the oracle over two steps."""
    import os
    case = 0
    for n in SWEEP_SIZES:
        for mis in range(8):
            gas = 1 + case % 3
            sizes = [n] if mode == "flat" else [n, 5]
            wl = workloads.custom(600 + case, sizes, decay=[True, False][:len(sizes)], gas=gas, steps=2,
                                  grad_sigma=0.3, misalign=mis, mode=mode)
            for pipe in ("0", "1"):
                os.environ["BF16OPT_PIPE"] = pipe
                try:
                    dense_parity(wl, defer=bool(case % 2))
                except AssertionError as e:
                    raise AssertionError(f"n={n} misalign={mis} gas={gas} defer={bool(case % 2)} "
                                         f"pipe={pipe}: {e}") from None
                finally:
                    os.environ.pop("BF16OPT_PIPE", None)
            case += 1


def _tiny_gradient_workload():
    """Gradients of magnitude 1e-25 ... 1e-18 (random sign, log-uniform), so
    that (1 - b2) g^2 spans FP32's subnormal range and underflow to zero while
    m stays normal; the norm is far below 1, so nothing is clipped."""
    wl = workloads.custom(295, [40_001, 99], decay=[True, False], gas=2, steps=3, grad_sigma=0.1, misalign=1)
    rng = np.random.default_rng(295)
    grads = []
    for _ in range(wl.steps * wl.gas):
        mag = 10.0 ** rng.uniform(-25, -18, wl.n)
        x = (mag * rng.choice([-1.0, 1.0], wl.n)).astype(np.float32)
        grads.append((x.view(np.uint32) >> 16).astype(np.uint16))       # bf16 by truncation
    return wl, grads


@needs_cuda
def test_gradients_with_subnormal_second_moments():
    import harness
    wl, grads = _tiny_gradient_workload()
    sh = GpuShard(wl, defer=True)
    for s in range(wl.steps):
        for k in range(wl.gas):
            sh.gbuf.copy_(torch.from_numpy(grads[s * wl.gas + k].view(np.int16)))
            sh.opt.accumulate(sh.grads_arg(), first=k == 0, last=k == wl.gas - 1, defer=k == wl.gas - 1)
        sh.opt.grad_norm(sync=True)
        sh.opt.step()
    torch.cuda.synchronize()
    got = sh.states()
    sh.close()

    p0 = synth.fill_master(wl, np.empty(wl.n, np.float32))
    p, m, v = p0.copy(), np.zeros(wl.n, np.float32), np.zeros(wl.n, np.float32)
    sc = {"M": np.zeros(wl.n), "A": np.abs(p0.astype(np.float64))}
    gof = wl.group_of(np.arange(wl.n))
    for s in range(wl.steps):
        ref = oracle.run_dense(p, lambda st, k: grads[s * wl.gas + k], wl.ranges(), ogroups(wl), 1, wl.gas,
                               wl.max_norm, t0=s, m=m, v=v)
        p, m, v = ref["p"], ref["m"], ref["v"]
        harness._update_scales(sc, wl, gof, ref["acc"], ref["clip"][0], m, v, s + 1, 1.0)
    tiny = np.finfo(np.float32).tiny
    assert np.count_nonzero((ref["v"] > 0) & (ref["v"] < tiny)) > 1000          # the case really is subnormal
    compare(got, ref, sc, wl, check_acc=False)


def _group(lr=6e-5, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.01):
    return dict(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay)


HYPER_EDGES = {
    # name: (groups for [decay, no-decay], max_norm, grad_scale)
    "clipping_off": ([_group(), _group(weight_decay=0.0)], 0.0, 1.0),
    "lr_zero": ([_group(lr=0.0), _group(lr=0.0, weight_decay=0.0)], 1.0, 1.0),
    "betas_zero": ([_group(beta1=0.0, beta2=0.0), _group(beta1=0.0, beta2=0.0, weight_decay=0.0)], 1.0, 1.0),
    "strong_decay": ([_group(lr=0.5, weight_decay=1.0), _group(lr=0.5, weight_decay=0.0)], 1.0, 1.0),
    "eps_one": ([_group(eps=1.0), _group(eps=1.0, weight_decay=0.0)], 1.0, 1.0),
    "negative_grad_scale": ([_group(), _group(weight_decay=0.0)], 1.0, -0.5),
}


@needs_cuda
@pytest.mark.parametrize("edge", sorted(HYPER_EDGES))
def test_hyper_parameter_edges(edge):
    """Clipping disabled (max_norm <= 0), lr = 0, beta1 = beta2 = 0 (no
    momentum, v = gc^2), weight decay 1 at lr 0.5, eps = 1 and a negative
    grad_scale: each equals the oracle over two steps (gradients large enough
    that clipping is active wherever it is on)."""
    groups, max_norm, gscale = HYPER_EDGES[edge]
    wl = workloads.custom(300 + sorted(HYPER_EDGES).index(edge), [30_000, 77, 5_000], decay=[True, False, True],
                          gas=2, steps=2, grad_sigma=0.5, misalign=1, max_norm=max_norm)
    wl.groups = groups
    dense_parity(wl, defer=True, grad_scale=gscale)


@needs_cuda
@pytest.mark.parametrize("mode", ["flat", "list"])
def test_sixteen_groups(mode):
    """The maximum of 16 parameter groups, each with its own lr, betas, eps and
    weight decay, over 16 tensors (group g = tensor g)."""
    rng = np.random.default_rng(16)
    wl = workloads.custom(320 + (mode == "list"), [int(x) for x in rng.integers(1, 9000, 16)], gas=2, steps=2,
                          grad_sigma=0.2, misalign=2, mode=mode)
    for g, t in enumerate(wl.tensors):
        t.group = g
    wl.groups = [_group(lr=float(10.0 ** rng.uniform(-5, -2)), beta1=float(rng.uniform(0.5, 0.99)),
                        beta2=float(rng.uniform(0.9, 0.999)), eps=float(10.0 ** rng.uniform(-9, -6)),
                        weight_decay=float(rng.choice([0.0, 0.01, 0.1]))) for _ in range(16)]
    dense_parity(wl, defer=True)


@needs_cuda
def test_two_handles_on_two_streams_interleaved():
    """Two independent shards (different layouts, sizes, GAS and deferral)
    driven at the same time on two non-blocking streams, their calls
    interleaved micro-batch by micro-batch: each equals the oracle, so handles
    share no state."""
    wa = workloads.custom(330, [70_001, 3], decay=[True, False], gas=3, steps=2, grad_sigma=0.2, misalign=1)
    wb = workloads.custom(331, [9_000, 12_345, 7], decay=[False, True, True], gas=2, steps=2, grad_sigma=0.05,
                          misalign=3, mode="list")
    A, B = GpuShard(wa, defer=[False, True, True]), GpuShard(wb, defer=True)
    torch.cuda.synchronize()                 # initial state written on the default stream
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for s in range(2):
        for k in range(max(wa.gas, wb.gas)):
            for sh, wl, st in ((A, wa, sa), (B, wb, sb)):
                if k < wl.gas:
                    buf = sh.gbufs[k % len(sh.gbufs)]
                    sgpu.fill_grad(wl, s, k, buf, stream=st)
                    sh.opt.accumulate(sh.grads_arg(buf), first=k == 0, last=k == wl.gas - 1,
                                      defer=sh.pattern[k], stream=st)
        for sh, st in ((A, sa), (B, sb)):
            sh.opt.grad_norm(stream=st)
        for sh, st in ((A, sa), (B, sb)):
            sh.opt.step(stream=st)
    torch.cuda.synchronize()
    for sh, wl in ((A, wa), (B, wb)):
        got = sh.states()
        sh.close()
        ref, scales = oracle_dense(wl, wl.steps)
        compare(got, ref, scales, wl, check_acc=not sh.defer)


@needs_cuda
def test_fast_pinned_buffers():
    """Rate-selected pinned host buffers: the requested count, pinned, with a
    measured rate each, and data that round-trips."""
    from host_buffers import fast_pinned_buffers
    n = 5_000_003
    dst = torch.empty(n, dtype=torch.int16, device="cuda")
    bufs, rates, rejected = fast_pinned_buffers(n, 2, dst, max_extra=2)
    assert len(bufs) == 2 and len(rates) == 2 and 0 <= rejected <= 2
    assert all(r > 0 for r in rates) and rates == sorted(rates, reverse=True)
    src = torch.randint(-30000, 30000, (n,), dtype=torch.int16, device="cuda")
    for hb in bufs:
        assert hb.tensor.is_pinned() and hb.tensor.numel() == n
        hb.tensor.copy_(src)
        dst.copy_(hb.tensor, non_blocking=True)
        torch.cuda.synchronize()
        assert torch.equal(dst, src)
        hb.close()


@needs_cuda
def test_claimed_chunks_on_a_full_chunk_shard(monkeypatch):
    """A shard of 2^25 + 4099 elements (full 32,768-element chunks, so its CTAs
    claim chunks, and its fused step runs the bulk-copy pipeline, by default)
    over many passes -- every deferral pattern the bench uses, two steps each --
    equals the fixed-stride schedule and the vector-load step bit for bit and
    the oracle within the tolerance."""
    wl = workloads.custom(280, [(1 << 25) - 1000, 5099], decay=[True, False], gas=4, steps=2, grad_sigma=0.01,
                          misalign=3)
    outs = []
    for sched, pipe in (("claim", "1"), ("static", "1"), ("claim", "0"), ("static", "0")):
        monkeypatch.setenv("BF16OPT_SCHEDULE", sched)
        monkeypatch.setenv("BF16OPT_PIPE", pipe)
        for pat in ([False, False, False, True], [True] * 4, [True, False, True, True]):
            sh = GpuShard(wl, defer=pat)
            sh.run(wl.steps)
            outs.append((sched, pat, sh.states(), list(sh.norms)))
            sh.close()
    for sched, pat, st, nr in outs[1:]:
        assert nr == outs[0][3], (sched, pat)
        for k in ("p", "m", "v", "p_bf16"):
            assert np.array_equal(st[k].view(np.uint8), outs[0][2][k].view(np.uint8)), (sched, pat, k)
    ref, scales = oracle_dense(wl, wl.steps)
    check_norms(outs[0][3], ref["sumsq"])
    compare(outs[0][2], ref, scales, wl, check_acc=False)
