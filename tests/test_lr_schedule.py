"""Learning-rate schedule (warmup + cosine decay to min_lr).

Source: "单机多卡实战：Megatron-DeepSpeed训练类BLOOM模型全流程解析", section 3
(lr 6e-5, min_lr 1e-6, lr_decay_style cosine, warmup_iters 500) and section 4
(--train-iters 100000).  The oracle's schedule is pinned by closed forms; the
library's host function is checked against the oracle (no GPU needed); the
GPU test steps a shard through warmup and decay.
"""
import math

import numpy as np
import pytest

import oracle
from mixed_precision_optimizer_bf16_gb300 import bf16opt as C
from mixed_precision_optimizer_bf16_gb300 import build as B

LR, MIN_LR, W, D = 6e-5, 1e-6, 500, 100_000


def test_oracle_schedule_closed_forms():
    f = lambda t: oracle.lr_at(LR, MIN_LR, W, D, t)
    assert f(1) == LR / 500
    assert f(250) == LR / 2
    assert f(500) == LR
    mid = W + (D - W) // 2                      # cos(pi/2) = 0: halfway between lr and min_lr
    assert f(mid) == pytest.approx(MIN_LR + (LR - MIN_LR) / 2, rel=1e-15)
    q = W + (D - W) // 4                        # cos(pi/4) = sqrt(2)/2
    assert f(q) == pytest.approx(MIN_LR + (LR - MIN_LR) * (1 + math.sqrt(0.5)) / 2, rel=1e-15)
    assert f(D) == MIN_LR                       # cos(pi) = -1
    assert f(D + 1) == MIN_LR and f(10 * D) == MIN_LR
    dec = [f(t) for t in range(W, D + 1, 997)]
    assert all(a >= b for a, b in zip(dec, dec[1:]))     # non-increasing after warmup
    assert f(W + 1) < LR and f(W + 1) > LR * (1 - 1e-8)


def test_library_factor_matches_oracle():
    B.build()
    s = C.lr_schedule(W, D, MIN_LR / LR)
    r = float(np.float32(MIN_LR / LR))
    for t in [1, 2, 3, 100, 499, 500, 501, 502, 1000, 25_000, 50_250, 75_000, 99_999, 100_000, 100_001, 10 ** 7]:
        rc, fac = C.bf16opt_lr_factor(s, t)
        assert rc == 0
        want = oracle.lr_at(1.0, r, W, D, t)
        assert abs(fac - want) <= 1e-15 * max(1.0, want), (t, fac, want)
    # degenerate schedules
    assert C.bf16opt_lr_factor(C.lr_schedule(0, 0, 0.5), 1) == (0, 0.5)
    assert C.bf16opt_lr_factor(C.lr_schedule(3, 3, 0.5), 3) == (0, 1.0)
    assert C.bf16opt_lr_factor(C.lr_schedule(3, 3, 0.5), 4) == (0, 0.5)
    assert C.bf16opt_lr_factor(C.lr_schedule(0, 10, 0.0), 10) == (0, 0.0)


@pytest.mark.parametrize("bad", [(10, 5, 0.1), (-1, 5, 0.1), (0, 5, -0.1), (0, 5, 1.5)])
def test_library_rejects_bad_schedules(bad):
    B.build()
    assert C.bf16opt_lr_factor(C.lr_schedule(*bad), 1)[0] == C.BF16OPT_ERR_INVALID_ARG
    assert C.bf16opt_lr_factor(C.lr_schedule(0, 5, 0.1), 0)[0] == C.BF16OPT_ERR_INVALID_ARG


@pytest.mark.gpu
def test_schedule_drives_the_step_on_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import synth
    import harness
    from synth import workloads
    wl = workloads.custom(210, [30_000, 777], decay=[True, False], gas=2, steps=6, grad_sigma=0.2)
    w, d, r = 2, 5, 0.25
    sh = harness.GpuShard(wl)
    sh.opt.set_lr_schedule(w, d, r)
    sh.run(wl.steps)
    got = sh.states()
    sh.close()
    # oracle with the schedule's absolute lr per step
    n = wl.n
    G = harness.ogroups(wl)
    gof = wl.group_of(np.arange(n))
    p = synth.fill_master(wl, np.empty(n, np.float32))
    sc = {"M": np.zeros(n), "A": np.abs(p.astype(np.float64))}
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    gfn = lambda s, k: synth.fill_grad(wl, s, k, np.empty(n, np.uint16))
    base = [dict(g) for g in wl.groups]
    rf = float(np.float32(r))
    for s in range(wl.steps):
        Gs = [oracle.group(oracle.lr_at(g.lr, g.lr * rf, w, d, s + 1), g.beta1, g.beta2, g.eps, g.weight_decay)
              for g in G]
        res = oracle.run_dense(p, gfn, wl.ranges(), Gs, 1, wl.gas, wl.max_norm, t0=s, m=m, v=v)
        p, m, v = res["p"], res["m"], res["v"]
        wl.groups = [dict(b, lr=gs.lr) for b, gs in zip(base, Gs)]
        harness._update_scales(sc, wl, gof, res["acc"], res["clip"][0], m, v, s + 1, 1.0)
    harness.compare(got, res, sc, wl)
