"""The seeded input generators (harness only): their values follow the input
recipe -- ~N(0, sigma) Irwin-Hall gradients truncated to bf16, a fixed 1 %
of exact zeros, log-uniform masters over 2^-26 ... 2^10 with random sign,
constant LayerNorm values -- and any element regenerates alone, bit for bit."""
import numpy as np

import synth
from synth import workloads


def _f32(bits16):
    return (bits16.astype(np.uint32) << 16).view(np.float32)


def test_gradient_moments_and_support():
    wl = workloads.workload(2)                       # sigma 1e-4
    g = _f32(synth.fill_grad(wl, 0, 0, np.empty(1 << 20, np.uint16), first=123_456_789)).astype(np.float64)
    s = wl.grad_sigma
    assert abs(g.mean()) < 5 * s / np.sqrt(g.size)
    assert abs(g.std() / s - 1.0) < 0.01             # truncation to bf16 shrinks |x| by < 2^-8
    assert np.abs(g).max() <= 3.47 * s               # Irwin-Hall(4) support: +-3.46 sigma


def test_forced_zeros_are_one_percent_and_fixed():
    wl = workloads.workload(5)                       # 1 % exact zeros
    n = 1 << 20
    a = synth.fill_grad(wl, 0, 0, np.empty(n, np.uint16))
    b = synth.fill_grad(wl, 3, 1, np.empty(n, np.uint16))
    za, zb = a == 0, b == 0
    assert abs(za.mean() - 0.01) < 0.001
    # the forced positions are shared by every micro-batch and step; besides
    # them a value is exactly 0 only when its Irwin-Hall sum is (about 1e-5)
    assert abs((za & zb).mean() - 0.01) < 0.001
    assert (za ^ zb).mean() < 1e-4


def test_loguniform_masters():
    wl = workloads.workload(5)
    p = synth.fill_master(wl, np.empty(1 << 20, np.float32))
    a = np.abs(p)
    assert a.min() >= 2.0 ** -26 and a.max() < 2.0 ** 10
    assert abs((p > 0).mean() - 0.5) < 0.005
    e = np.floor(np.log2(a)).astype(int)
    counts = np.bincount(e + 26, minlength=36)
    assert counts.min() > 0.9 * a.size / 36 and counts.max() < 1.1 * a.size / 36   # octaves uniform


def test_constant_layernorm_masters():
    wl = workloads.workload(2)
    names = [t.name for t in wl.tensors]
    gi = names.index("h.0.ln1.gamma")
    bi = names.index("h.0.ln1.beta")
    g = synth.fill_master(wl, np.empty(wl.tensors[gi].numel, np.float32), wl.offsets[gi])
    b = synth.fill_master(wl, np.empty(wl.tensors[bi].numel, np.float32), wl.offsets[bi])
    assert np.all(g == 1.0) and np.all(b == 0.0)


def test_gather_equals_fill():
    wl = workloads.workload(5)
    n = 200_000
    full_g = synth.fill_grad(wl, 2, 1, np.empty(n, np.uint16))
    full_p = synth.fill_master(wl, np.empty(n, np.float32))
    idx = np.random.default_rng(0).integers(0, n, 5000)
    assert np.array_equal(synth.gather_grad(wl, 2, 1, idx), full_g[idx])
    assert np.array_equal(synth.gather_master(wl, idx).view(np.uint32), full_p[idx].view(np.uint32))


def test_streams_are_independent():
    wl = workloads.workload(1)
    n = 1 << 18
    x = [_f32(synth.fill_grad(wl, s, k, np.empty(n, np.uint16))).astype(np.float64)
         for s, k in ((0, 0), (0, 1), (1, 0))]
    for i in range(3):
        for j in range(i + 1, 3):
            assert abs(np.corrcoef(x[i], x[j])[0, 1]) < 0.01
