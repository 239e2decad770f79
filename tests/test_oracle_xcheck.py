"""Cross-checks of the CPU oracle against independent implementations (no GPU).

* A brute-force re-evaluation in 50-digit decimal arithmetic of whole steps
  (accumulate, global norm, clip, AdamW, bf16), rounded to FP32 by an exact
  rational routine, on tiny inputs with two parameter groups.
* torch.optim.AdamW (float64, CPU, foreach=False) as the library special case,
  with the clip applied to the gradient by hand and FP32 re-storage per step.
* The streamed (regenerate-from-counters) oracle entry points against the
  materialised ones.
"""
from decimal import Decimal
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from synth import workloads
from exact import D, f32_bits, rn32, rne_bf16_bits_from_f32

LR, B1, B2, EPS, WD = 6e-5, 0.9, 0.95, 1e-8, 0.01


def _dec_rn32(d):
    return Decimal(rn32(Fraction(d))[0])


def decimal_run(p0, grads, ranges, wds, steps, gas, max_norm):
    """Whole-run brute force in Decimal (50 digits); storage points rounded to FP32."""
    n = len(p0)
    p = [D(x) for x in p0]
    m = [Decimal(0)] * n
    v = [Decimal(0)] * n
    b1, b2, eps, lr = D(B1), D(B2), D(EPS), D(LR)
    accs = None
    for s in range(steps):
        acc = [Decimal(0)] * n
        for k in range(gas):
            g = [D(x) for x in oracle.bf16_to_f32(grads[s][k])]
            acc = [g[i] if k == 0 else _dec_rn32(acc[i] + g[i]) for i in range(n)]
        S = sum(a * a for a in acc)
        norm = S.sqrt()
        c = D(max_norm) / norm if norm > D(max_norm) else Decimal(1)
        t = s + 1
        bc1 = 1 - b1 ** t
        bc2 = 1 - b2 ** t
        for b, e, gi in ranges:
            wd = D(wds[gi])
            for i in range(b, e):
                gc = acc[i] * c
                m1 = b1 * m[i] + (1 - b1) * gc
                v1 = b2 * v[i] + (1 - b2) * gc * gc
                mh, vh = m1 / bc1, v1 / bc2
                p1 = p[i] - lr * wd * p[i] - lr * mh / (vh.sqrt() + eps)
                m[i], v[i], p[i] = _dec_rn32(m1), _dec_rn32(v1), _dec_rn32(p1)
        accs = acc
    return p, m, v, accs


@pytest.mark.parametrize("n,gas,steps,sigma", [(64, 3, 3, 0.5), (17, 1, 2, 1e-3), (40, 2, 3, 3.0)])
def test_decimal_brute_force(n, gas, steps, sigma):
    rng = np.random.default_rng(n * 100 + gas)
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    grads = [[oracle.f32_to_bf16(rng.normal(0, sigma, n).astype(np.float32)) for _ in range(gas)]
             for _ in range(steps)]
    ranges = [(0, n // 3, 0), (n // 3, n // 2, 1), (n // 2, n, 0)]
    wds = [WD, 0.0]
    groups = [oracle.group(LR, B1, B2, EPS, WD), oracle.group(LR, B1, B2, EPS, 0.0)]
    res = oracle.run_dense(p0.copy(), lambda s, k: grads[s][k], ranges, groups, steps, gas, 1.0, threads=2)
    pd, md, vd, accd = decimal_run(p0, grads, ranges, wds, steps, gas, 1.0)
    for got, want in ((res["p"], pd), (res["m"], md), (res["v"], vd), (res["acc"], accd)):
        assert [f32_bits(x) for x in got] == [f32_bits(np.float32(float(w))) for w in want]
    assert res["p_bf16"].tolist() == [rne_bf16_bits_from_f32(x) for x in res["p"]]
    # the largest case really clips
    if sigma >= 0.5:
        assert res["clip"][0] < 1.0


def test_torch_adamw_library_case():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    n, steps = 1_000_000, 3
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    accs = [(rng.normal(0, 5e-4, n) * (40.0 if s == 1 else 1.0)).astype(np.float32) for s in range(steps)]
    # oracle
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    pb = np.zeros(n, np.uint16)
    G = oracle.group(LR, B1, B2, EPS, WD)
    clips = []
    for s in range(steps):
        c = oracle.clip_coef(oracle.sumsq(accs[s]), 1.0)
        clips.append(c)
        oracle.adamw(p, m, v, pb, accs[s], c, G, s + 1)
    assert clips[1] < 1.0 and clips[0] == 1.0
    # torch, float64, manual clip, FP32 re-storage
    tp = torch.nn.Parameter(torch.from_numpy(p0.astype(np.float64)))
    opt = torch.optim.AdamW([tp], lr=LR, betas=(B1, B2), eps=EPS, weight_decay=WD, foreach=False)
    for s in range(steps):
        tp.grad = torch.from_numpy(accs[s].astype(np.float64)) * clips[s]
        opt.step()
        with torch.no_grad():
            tp.copy_(tp.float().double())
            st = opt.state[tp]
            st["exp_avg"].copy_(st["exp_avg"].float().double())
            st["exp_avg_sq"].copy_(st["exp_avg_sq"].float().double())
    st = opt.state[tp]
    for mine, theirs in ((p, tp.detach()), (m, st["exp_avg"]), (v, st["exp_avg_sq"])):
        t32 = theirs.float().numpy()
        d = np.abs(mine.view(np.int32).astype(np.int64) - t32.view(np.int32).astype(np.int64))
        assert d.max() <= 1


def test_stream_sumsq_matches_dense():
    wl = workloads.custom(901, [70_001, 3, 65_536, 129], gas=3, grad_sigma=2e-3, zero_frac=0.05)
    st = oracle.stream(wl.id, wl.gas, synth.sigma_scale(wl.grad_sigma), synth.zero_thresh(wl.zero_frac))
    for step in (0, 1):
        acc = np.zeros(wl.n, np.float32)
        for k in range(wl.gas):
            g = synth.fill_grad(wl, step, k, np.empty(wl.n, np.uint16))
            oracle.accumulate(acc, g, first=(k == 0))
        assert oracle.stream_sumsq(st, step, wl.n, threads=3) == oracle.sumsq(acc)


def test_sample_run_matches_dense():
    wl = workloads.custom(902, [1000, 37, 5000], decay=[True, False, True], gas=2, steps=3, grad_sigma=0.3)
    n = wl.n
    st = oracle.stream(wl.id, wl.gas, synth.sigma_scale(wl.grad_sigma))
    groups = [oracle.group(**g) for g in wl.groups]
    p0 = synth.fill_master(wl, np.empty(n, np.float32))
    res = oracle.run_dense(p0.copy(), lambda s, k: synth.fill_grad(wl, s, k, np.empty(n, np.uint16)),
                           wl.ranges(), groups, wl.steps, wl.gas, wl.max_norm)
    assert res["clip"][0] < 1.0
    idx = np.array([0, 1, 999, 1000, 1036, 1037, 6036], np.uint64)
    p, m, v, pb, acc = oracle.sample_run(st, idx, p0[idx.astype(np.int64)], groups, wl.group_of(idx),
                                         res["clip"])
    ii = idx.astype(np.int64)
    assert np.array_equal(p, res["p"][ii]) and np.array_equal(m, res["m"][ii])
    assert np.array_equal(v, res["v"][ii]) and np.array_equal(pb, res["p_bf16"][ii])
    assert np.array_equal(acc, res["acc"][ii])
