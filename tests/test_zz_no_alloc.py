"""The allocation-free norm entry point (bf16opt_grad_norm_static).

It serves callers that cannot call cudaMalloc (code inside another
framework's launch path that only gets a stream, processes whose device
memory sits in a caching allocator, loops that cannot take the device
synchronisation of cudaMalloc/cudaFree): its scratch is a fixed static device
array.  This file is collected last so that a run stopping at its first
failure has already run every other test; it must pass alone in a fresh
process as well as after the other tests.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from mixed_precision_optimizer_bf16_gb300 import bf16opt as C  # noqa: E402
from mixed_precision_optimizer_bf16_gb300.optimizer import BF16Optimizer, alloc_flat  # noqa: E402
from synth import gpu as sgpu, workloads  # noqa: E402

pytestmark = pytest.mark.gpu

REL = 1e-6  # the norm tolerance of the parity tests


def _read(res):
    h = res.cpu().numpy().view(np.float64)
    return float(h[0]), float(h[1]), float(h[2])


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_static_norm_matches_handle_norm_twice():
    """Two calls in a row on the same accumulator give the handle's own sum of
    squares bit for bit (the same chunking, thread map and fixed-order sums),
    and the oracle's FP64 sum of squares of the copied-back accumulator within
    the norm tolerance."""
    C.load()
    # 3,000,011 elements (ragged last chunk), misaligned by 1 element, clipping active
    wl = workloads.custom(199, [3_000_011], gas=2, steps=1, grad_sigma=0.05, misalign=1)
    flat = alloc_flat(wl.n, "cuda", wl.misalign)
    sgpu.fill_master(wl, flat["master"])
    for k in ("exp_avg", "exp_avg_sq", "grad_accum", "param_bf16"):
        flat[k].zero_()
    g = torch.empty(wl.n + 64, dtype=torch.int16, device="cuda")[1:1 + wl.n]
    opt = BF16Optimizer(wl.groups, flat=flat, max_grad_norm=1.0, grad_scale=0.5)
    for k in range(2):
        sgpu.fill_grad(wl, 0, k, g)
        opt.accumulate(g, first=k == 0, last=k == 1)
    stream = torch.cuda.current_stream().cuda_stream
    rc, handle_sumsq = C.bf16opt_grad_norm_local(opt.h, stream)
    assert rc == 0
    acc = flat["grad_accum"]
    ref_sumsq = oracle.sumsq(acc.cpu().numpy(), 0.5)
    ref_norm = math.sqrt(ref_sumsq)
    assert ref_norm > 1.0  # clipping is active

    res = torch.zeros(3, dtype=torch.float64, device="cuda")   # caller-owned output
    outs = []
    for _ in range(2):  # two calls in a row share the static scratch
        rc = C.bf16opt_grad_norm_static(acc.data_ptr(), acc.numel(), 0.5, 1.0, res.data_ptr(), stream)
        assert rc == 0, C.bf16opt_last_error(None)
        torch.cuda.synchronize()
        outs.append(_read(res))
        res.zero_()
    for sumsq, norm, clip in outs:
        assert sumsq == handle_sumsq                        # the handle's reduction, bit for bit
        assert norm == math.sqrt(handle_sumsq) and clip == 1.0 / norm
        assert abs(sumsq - ref_sumsq) <= REL * ref_sumsq    # and the oracle's sum
        assert abs(norm - ref_norm) <= REL * ref_norm
        assert abs(clip - 1.0 / ref_norm) <= REL / ref_norm
    assert outs[0] == outs[1]

    # a smaller second input right after a larger one: no stale partial is used
    part = acc[:70_000]
    rc = C.bf16opt_grad_norm_static(part.data_ptr(), part.numel(), 1.0, 1.0, res.data_ptr(), stream)
    assert rc == 0
    torch.cuda.synchronize()
    s_small = oracle.sumsq(part.cpu().numpy())
    assert abs(_read(res)[0] - s_small) <= REL * s_small

    # empty input and the size limit
    assert C.bf16opt_grad_norm_static(0, 0, 1.0, 1.0, res.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    assert _read(res) == (0.0, 0.0, 1.0)
    too_big = C.BF16OPT_STATIC_NORM_MAX_ELEMS + 1
    assert C.bf16opt_grad_norm_static(acc.data_ptr(), too_big, 1.0, 1.0, res.data_ptr(), stream) == \
        C.BF16OPT_ERR_INVALID_ARG
    assert "exceeds" in C.bf16opt_last_error(None)
    opt.close()


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_static_norm_refuses_memory_the_device_cannot_use():
    """The kernels write `out` and read `grad_accum` directly, so ordinary
    (pageable) host memory is refused with an error instead of being handed to
    a kernel; page-locked host memory works through its mapped address."""
    C.load()
    stream = torch.cuda.current_stream().cuda_stream
    acc = torch.full((100_003,), 0.25, dtype=torch.float32, device="cuda")
    res = torch.zeros(3, dtype=torch.float64, device="cuda")
    host_out = np.zeros(3, np.float64)
    host_acc = np.full(100_003, 0.25, np.float32)
    assert C.bf16opt_grad_norm_static(acc.data_ptr(), acc.numel(), 1.0, 1.0, host_out.ctypes.data, stream) == \
        C.BF16OPT_ERR_INVALID_ARG
    assert "out must be" in C.bf16opt_last_error(None)
    assert C.bf16opt_grad_norm_static(host_acc.ctypes.data, host_acc.size, 1.0, 1.0, res.data_ptr(), stream) == \
        C.BF16OPT_ERR_INVALID_ARG
    assert "grad_accum must be" in C.bf16opt_last_error(None)
    assert host_out.tolist() == [0.0, 0.0, 0.0]
    pinned = torch.zeros(3, dtype=torch.float64, pin_memory=True)
    assert C.bf16opt_grad_norm_static(acc.data_ptr(), acc.numel(), 1.0, 1.0, pinned.data_ptr(), stream) == 0
    assert C.bf16opt_grad_norm_static(acc.data_ptr(), acc.numel(), 1.0, 1.0, res.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    want = 100_003 * 0.0625
    assert tuple(pinned.tolist()) == _read(res) and pinned[0].item() == want


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_static_norm_of_values_whose_squares_overflow_fp32():
    """FP32 accumulator values of 1.5e19 ... 3e30 are finite but their squares
    are not in FP32; the norm is the FP64 sum of squares (each square of an
    FP32 value is exact in FP64; math.fsum rounds the sum once).  Values sit in
    the head, the vector body and the tail of the chunks.  An infinite element
    gives an infinite norm and a zero clip coefficient, a NaN one a NaN norm."""
    C.load()
    rng = np.random.default_rng(5)
    n = 200_003
    host = rng.normal(0.0, 0.1, n).astype(np.float32)
    for i, x in {0: 1.5e19, 3: -2e20, 70_000: 3e30, 70_001: -1e25, n - 1: 7e21}.items():
        host[i] = x
    acc = torch.empty(n + 64, dtype=torch.float32, device="cuda")[3:3 + n]
    acc.copy_(torch.from_numpy(host))
    res = torch.zeros(3, dtype=torch.float64, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert C.bf16opt_grad_norm_static(acc.data_ptr(), n, 1.0, 1.0, res.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    sumsq, norm, clip = _read(res)
    ref = math.fsum(float(x) * float(x) for x in host.tolist())
    assert abs(oracle.sumsq(host) - ref) <= 1e-15 * ref
    assert abs(sumsq - ref) <= REL * ref
    assert abs(norm - math.sqrt(ref)) <= REL * math.sqrt(ref)
    assert abs(clip - 1.0 / math.sqrt(ref)) <= REL / math.sqrt(ref)

    acc[5] = float("inf")
    assert C.bf16opt_grad_norm_static(acc.data_ptr(), n, 1.0, 1.0, res.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    sumsq, norm, clip = _read(res)
    assert math.isinf(norm) and norm > 0 and clip == 0.0
    acc[7] = float("nan")
    assert C.bf16opt_grad_norm_static(acc.data_ptr(), n, 1.0, 1.0, res.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    assert math.isnan(_read(res)[1])
