"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test states what pins it: a closed form, an invariant, a textbook or
library routine, exact/brute-force arithmetic, or a hand-computed value.  The
method's definition comes from "BLOOM 176B 训练技术概览" (section "BF16 优化器":
FP32 accumulation across micro-batches), "企业官网建设流程全解析" (cf-1.com,
sections 1, 3.3 and 4.3: FP32 master/momentum/variance, AdamW lr 6e-5 wd 0.01,
global-norm clipping at 1.0) and "单机多卡实战：Megatron-DeepSpeed训练类BLOOM模型全流程解析"
(section 3: GAS 4, clip_grad 1.0).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from exact import F, adam_bound, bits_f32, f32_bits, rn32, rn32_bits, rne_bf16_bits_from_f32

LR, B1, B2, EPS, WD = 6e-5, 0.9, 0.95, 1e-8, 0.01


def grp(wd=WD, lr=LR, b1=B1, b2=B2, eps=EPS):
    return oracle.group(lr, b1, b2, eps, wd)


def one_step(p0, g_acc, t=1, c=1.0, wd=WD, m0=0.0, v0=0.0, grad_scale=1.0):
    p = np.array(p0, np.float32).reshape(-1).copy()
    m = np.full(p.size, m0, np.float32)
    v = np.full(p.size, v0, np.float32)
    pb = np.zeros(p.size, np.uint16)
    acc = np.array(g_acc, np.float32).reshape(-1).copy()
    oracle.adamw(p, m, v, pb, acc, c, grp(wd), t, grad_scale=grad_scale, threads=1)
    return p, m, v, pb


# --------------------------------------------------------------------- P1 cast

def test_bf16_cast_hand_values():
    """1 + 2^-8 is a tie between 1.0 and the next bf16 and goes to even (0x3F80);
    1 + 3*2^-8 ties between 0x3F81 and 0x3F82 and goes to even (0x3F82)."""
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8), 0.0, -0.0],
                 np.float32)
    got = oracle.f32_to_bf16(x)
    assert got.tolist() == [0x3F80, 0x3F82, 0x3F81, 0xBF80, 0x0000, 0x8000]
    h = oracle.f32_to_bf16(np.array([np.nan, np.inf, -np.inf, 3.4e38], np.float32))
    assert (h[0] & 0x7F80) == 0x7F80 and (h[0] & 0x7F) != 0
    assert h[1] == 0x7F80 and h[2] == 0xFF80 and h[3] == 0x7F80  # 3.4e38 rounds up to +inf


def test_bf16_cast_exact_neighbours():
    """Against an exact-rational choice between the two bf16 neighbours."""
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2 ** 32, 4000, dtype=np.uint64).astype(np.uint32)
    u[:64] = (u[:64] & 0xFFFF0000) | 0x8000  # exact ties
    f = u.view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) < 3.0e38)]
    got = oracle.f32_to_bf16(f)
    want = [rne_bf16_bits_from_f32(x) for x in f]
    assert got.tolist() == want


@pytest.mark.slow
def test_bf16_cast_exhaustive_vs_torch():
    """All 2^32 binary32 patterns against torch's CPU float->bfloat16 conversion
    (round to nearest even); NaNs must stay NaN."""
    torch = pytest.importorskip("torch")
    ch = 1 << 26
    for c in range(0, 1 << 32, ch):
        u = np.arange(c, c + ch, dtype=np.uint64).astype(np.uint32)
        f = u.view(np.float32)
        a = oracle.f32_to_bf16(f)
        b = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(f)
        assert np.array_equal(a[~nan], b[~nan])
        an = a[nan]
        assert np.all(((an & 0x7F80) == 0x7F80) & ((an & 0x7F) != 0))


# ------------------------------------------------------------- P2/P3 accumulate

def test_accumulate_tie_to_even():
    """bf16 grads [1.0, 2^-24] over two micro-batches: 1 + 2^-24 is the midpoint of
    1 and 1 + 2^-23, so the FP32 sum is exactly 1.0 (ties to even)."""
    acc = np.zeros(1, np.float32)
    oracle.accumulate(acc, oracle.f32_to_bf16(np.array([1.0], np.float32)), first=True)
    oracle.accumulate(acc, oracle.f32_to_bf16(np.array([2.0 ** -24], np.float32)), first=False)
    assert f32_bits(acc[0]) == 0x3F800000


def test_accumulate_matches_numpy_float32_adds():
    """FP32 storage after every micro-batch, in micro-batch order = numpy float32 adds."""
    rng = np.random.default_rng(2)
    n, G = 100_003, 5
    gs = [oracle.f32_to_bf16(rng.normal(0, 10.0 ** rng.integers(-8, 3), n).astype(np.float32)) for _ in range(G)]
    acc = np.full(n, 123.0, np.float32)
    for k in range(G):
        oracle.accumulate(acc, gs[k], first=(k == 0))
    ref = oracle.bf16_to_f32(gs[0]).copy()
    for k in range(1, G):
        ref = (ref + oracle.bf16_to_f32(gs[k])).astype(np.float32)
    assert np.array_equal(acc.view(np.uint32), ref.view(np.uint32))


def test_accumulate_is_sum_not_mean():
    """GAS micro-batches of the same gradient g give G*g (exact for small G)."""
    g = oracle.f32_to_bf16(np.array([0.75, -3.0, 2.0 ** -30], np.float32))
    acc = np.zeros(3, np.float32)
    for k in range(4):
        oracle.accumulate(acc, g, first=(k == 0))
    assert acc.tolist() == [3.0, -12.0, 4 * 2.0 ** -30]


# ------------------------------------------------------------------ norm, clip

def test_sumsq_vs_fsum_and_numpy_norm():
    """Sum of exact FP64 squares vs math.fsum (correctly rounded), within the
    recursive-summation bound, and vs numpy's 2-norm."""
    rng = np.random.default_rng(3)
    n = 300_001
    acc = rng.normal(0, 1e-3, n).astype(np.float32)
    S = oracle.sumsq(acc)
    sq = acc.astype(np.float64) ** 2
    exact = math.fsum(sq.tolist())
    gamma = (65536 + n // 65536 + 2) * 2.0 ** -53
    assert abs(S - exact) <= gamma * exact
    assert abs(math.sqrt(S) - np.linalg.norm(acc.astype(np.float64))) <= 1e-13 * math.sqrt(S)


def test_sumsq_copies_closed_form():
    """N copies of a: S = N a^2 exactly (a power of two), norm = |a| sqrt(N)."""
    for a, n in ((0.5, 1 << 20), (-2.0 ** -12, 12345), (3.0, 7)):
        acc = np.full(n, a, np.float32)
        assert oracle.sumsq(acc) == n * a * a


def test_sumsq_grad_scale_is_rounded_product():
    """With grad_scale s the norm sees RN32(acc * s) (numpy float32 multiply)."""
    rng = np.random.default_rng(4)
    acc = rng.normal(0, 1, 5000).astype(np.float32)
    s = np.float32(0.3)
    e = (acc * s).astype(np.float32).astype(np.float64)
    exact = math.fsum((e * e).tolist())
    assert abs(oracle.sumsq(acc, grad_scale=float(s)) - exact) <= (acc.size + 2) * 2.0 ** -53 * exact
    # and the unscaled sum differs by ~s^2 (the scale is really applied)
    assert oracle.sumsq(acc) * 0.09 == pytest.approx(exact, rel=1e-6)


def test_clip_coef_closed_forms():
    """norm <= max -> exactly 1; norm = C > max -> max/C; g = [3, 4] -> norm 5 -> 0.2."""
    assert oracle.clip_coef(0.25, 1.0) == 1.0
    assert oracle.clip_coef(1.0, 1.0) == 1.0          # norm == max_norm: unchanged
    assert oracle.clip_coef(25.0, 1.0) == 0.2
    assert oracle.clip_coef(25.0, 0.0) == 1.0         # clipping off
    assert oracle.clip_coef(4.0 * 7.0 ** 2, 1.0) == 1.0 / 14.0
    acc = np.array([3.0, 4.0], np.float32)
    assert oracle.clip_coef(oracle.sumsq(acc), 1.0) == 0.2


# ------------------------------------------------------------ AdamW closed forms

def test_step1_closed_form_random():
    """At t = 1 from m = v = 0: m_hat = gc and sqrt(v_hat) = |gc|, so
    p1 = p0 (1 - lr wd) - lr gc / (|gc| + eps), m1 = (1-b1) gc, v1 = (1-b2) gc^2,
    each rounded once to FP32.  Exact rationals, no square root needed."""
    rng = np.random.default_rng(5)
    n = 3000
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    acc = (rng.normal(0, 1e-3, n) * 10.0 ** rng.integers(-6, 2, n)).astype(np.float32)
    acc[:20] = 0.0
    c = 0.375
    p, m, v, pb = one_step(p0, acc, t=1, c=c)
    lr, wd, eps, b1, b2 = F(LR), F(WD), F(EPS), F(B1), F(B2)
    n_amb = 0
    for i in range(n):
        gc = F(acc[i]) * F(c)
        pe = F(p0[i]) - lr * wd * F(p0[i]) - lr * gc / (abs(gc) + eps)
        for got, want in ((p[i], pe), (m[i], (1 - b1) * gc), (v[i], (1 - b2) * gc * gc)):
            wb, dist = rn32_bits(want)
            if dist < Fraction(1, 2 ** 40):
                n_amb += 1
                assert abs(f32_bits(got) - wb) <= 1
            else:
                assert f32_bits(got) == wb, (i, got, float(want))
        assert pb[i] == rne_bf16_bits_from_f32(p[i])
    assert n_amb < 5


def test_hand_worked_single_element():
    """p0 = 1, g = 0.5, wd 0.01, t = 1:
    p1 = (1 - 6e-7) - 6e-5 * 0.5 / (0.5 + 1e-8) = 0.99993940000120 (exact),
    nearest FP32 = 1 - 1017 * 2^-24 = 0.99993938207626 (0x3F7FFC07);
    m1 = 0.05 -> 0x3D4CCCCD; v1 = 0.0125 -> 0x3C4CCCCD; bf16(p1) = 0x3F80."""
    p, m, v, pb = one_step([1.0], [0.5])
    assert f32_bits(p[0]) == 0x3F7FFC07
    assert f32_bits(m[0]) == 0x3D4CCCCD
    assert f32_bits(v[0]) == 0x3C4CCCCD
    assert pb[0] == 0x3F80


def test_hand_worked_two_steps():
    """The single-element case continued: g = -0.25 at t = 2 from the stored
    FP32 state of step 1.  Expected values from exact rationals (the square
    root in 50-digit decimal), each rounded once to FP32:
    m2 = 0.9 m1 - 0.025 -> 0x3CA3D70B, v2 = 0.95 v1 + 0.003125 -> 0x3C75C290,
    p2 = p1 (1 - lr wd) - lr m2/(1 - 0.9^2) / (sqrt(v2/(1 - 0.95^2)) + eps)
    -> 0x3F7FFAEF; bias correction at t = 2 is what moves it."""
    from decimal import Decimal
    p = np.array([1.0], np.float32)
    m = np.zeros(1, np.float32)
    v = np.zeros(1, np.float32)
    pb = np.zeros(1, np.uint16)
    oracle.adamw(p, m, v, pb, np.array([0.5], np.float32), 1.0, grp(), 1, threads=1)
    p1, m1, v1 = F(p[0]), F(m[0]), F(v[0])
    g = F(-0.25)
    oracle.adamw(p, m, v, pb, np.array([-0.25], np.float32), 1.0, grp(), 2, threads=1)

    m2 = F(B1) * m1 + (1 - F(B1)) * g
    v2 = F(B2) * v1 + (1 - F(B2)) * g * g
    vhat = v2 / (1 - F(B2) ** 2)
    root = Fraction((Decimal(vhat.numerator) / Decimal(vhat.denominator)).sqrt())
    p2 = p1 - F(LR) * F(WD) * p1 - F(LR) * (m2 / (1 - F(B1) ** 2)) / (root + F(EPS))
    for got, want in ((m[0], m2), (v[0], v2), (p[0], p2)):
        bits, mid = rn32_bits(want)
        assert mid > 1e-12
        assert f32_bits(got) == bits
    assert (f32_bits(m[0]), f32_bits(v[0]), f32_bits(p[0])) == (0x3CA3D70B, 0x3C75C290, 0x3F7FFAEF)
    assert pb[0] == rne_bf16_bits_from_f32(p[0]) == 0x3F80


def test_hand_worked_rounding_point_no_decay():
    """Accumulated grad exactly 1.0 (see the tie test), norm = 1 = max_norm so
    c = 1, wd = 0: p1 = 1 - 6e-5 / (1 + 1e-8) = 0.99994000000060, nearest FP32
    1 - 1007 * 2^-24 = 0x3F7FFC11; m1 = 0.1 -> 0x3DCCCCCD; v1 = 0.05 -> 0x3D4CCCCD."""
    c = oracle.clip_coef(oracle.sumsq(np.array([1.0], np.float32)), 1.0)
    assert c == 1.0
    p, m, v, pb = one_step([1.0], [1.0], c=c, wd=0.0)
    assert (f32_bits(p[0]), f32_bits(m[0]), f32_bits(v[0])) == (0x3F7FFC11, 0x3DCCCCCD, 0x3D4CCCCD)


def test_hand_worked_clip_3_4():
    """g = [3, 4]: norm 5, c = 0.2, gc = [0.6, 0.8]: m = RN32(0.06), RN32(0.08);
    v = RN32(0.018), RN32(0.032); p = 0x3F7FFC07 for both (step-1 update ~ lr)."""
    acc = np.array([3.0, 4.0], np.float32)
    c = oracle.clip_coef(oracle.sumsq(acc), 1.0)
    p, m, v, pb = one_step([1.0, 1.0], acc, c=c)
    assert [f32_bits(x) for x in m] == [0x3D75C28F, 0x3DA3D70A]
    assert [f32_bits(x) for x in v] == [0x3C9374BC, 0x3D03126F]
    assert [f32_bits(x) for x in p] == [0x3F7FFC07, 0x3F7FFC07]


def test_small_master_negative_grad():
    """p0 = RN32(0.02), g = -2^-10: the step moves p up by ~lr.  Exact rational
    closed form (t = 1), then one FP32 rounding."""
    p0 = np.float32(0.02)
    g = -(2.0 ** -10)
    p, m, v, pb = one_step([p0], [g])
    want = F(p0) - F(LR) * F(WD) * F(p0) - F(LR) * F(g) / (abs(F(g)) + F(EPS))
    assert f32_bits(p[0]) == rn32_bits(want)[0]
    assert f32_bits(m[0]) == rn32_bits((1 - F(B1)) * F(g))[0]
    assert pb[0] == rne_bf16_bits_from_f32(p[0])


def test_pure_decay_invariant():
    """g = 0, m = v = 0: m and v stay 0 and p_t = RN32(p_{t-1} (1 - lr wd));
    p0 = 0.5 gives 0x3EFFFFF6, 0x3EFFFFEC, 0x3EFFFFE2.  With wd = 0 nothing moves."""
    p = np.array([0.5, -3.0, 1e-30], np.float32)
    m = np.zeros(3, np.float32)
    v = np.zeros(3, np.float32)
    pb = np.zeros(3, np.uint16)
    acc = np.zeros(3, np.float32)
    ref = [F(x) for x in p]
    for t in (1, 2, 3):
        oracle.adamw(p, m, v, pb, acc, 1.0, grp(), t)
        ref = [Fraction(rn32(r * (1 - F(LR) * F(WD)))[0]) for r in ref]
        assert [f32_bits(x) for x in p] == [rn32_bits(r)[0] for r in ref]
        assert not m.any() and not v.any()
    assert [f32_bits(p[0])] == [0x3EFFFFE2]
    p2 = np.array([0.5, -3.0], np.float32)
    m2, v2, pb2 = np.zeros(2, np.float32), np.zeros(2, np.float32), np.zeros(2, np.uint16)
    for t in (1, 2, 3):
        oracle.adamw(p2, m2, v2, pb2, np.zeros(2, np.float32), 1.0, grp(wd=0.0), t)
    assert p2.tolist() == [0.5, -3.0]
    assert pb2.tolist() == [0x3F00, 0xC040]


def test_adam_step_bound_multi_step():
    """|p' - p (1 - lr wd)| <= lr * B_t (Cauchy-Schwarz bound on |m_hat/sqrt(v_hat)|),
    B = 1, 1.000364, 1.000969, 1.001811, 1.002884 for t = 1..5, up to rounding."""
    rng = np.random.default_rng(6)
    n = 20000
    p = rng.normal(0, 0.02, n).astype(np.float32)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    pb = np.zeros(n, np.uint16)
    expect_B = [1.0, 1.000364, 1.000969, 1.001811, 1.002884]
    for t in range(1, 6):
        assert adam_bound(t, B1, B2) == pytest.approx(expect_B[t - 1], abs=2e-6)
        acc = rng.standard_cauchy(n).astype(np.float32) * np.float32(1e-3)
        before = p.astype(np.float64)
        oracle.adamw(p, m, v, pb, acc, 1.0, grp(), t)
        dec = before * (1 - LR * WD)
        step = np.abs(p.astype(np.float64) - dec)
        bound = LR * adam_bound(t, B1, B2) * (1 + 1e-5) + np.abs(before) * 2.0 ** -23
        assert np.all(step <= bound)
        # and the bound is nearly attained somewhere (the update is not trivially small)
        assert step.max() > 0.9 * LR


def test_bias_correction_constant_gradient():
    """Constant gradient g every step: m_hat = g and v_hat = g^2 exactly in exact
    arithmetic for all t (bias correction undoes the zero start), so every step
    moves p by lr * |g|/(|g| + eps) toward -sign(g), plus decay."""
    g = 2.0 ** -9
    p = np.array([0.25], np.float32)
    m, v, pb = np.zeros(1, np.float32), np.zeros(1, np.float32), np.zeros(1, np.uint16)
    ref = F(p[0])
    for t in range(1, 8):
        oracle.adamw(p, m, v, pb, np.array([g], np.float32), 1.0, grp(), t)
        ref = Fraction(rn32(ref - F(LR) * F(WD) * ref - F(LR) * F(g) / (F(g) + F(EPS)))[0])
        assert abs(f32_bits(p[0]) - f32_bits(np.float32(float(ref)))) <= 1


def test_grad_scale_applies_before_clip_and_moments():
    """grad_scale s: the update sees RN32(acc * s); with s = 2 and acc = 0.25 the
    step equals the unscaled step on acc = 0.5."""
    a = one_step([1.0], [0.25], grad_scale=2.0)
    b = one_step([1.0], [0.5])
    assert [f32_bits(x[0]) for x in a[:3]] == [f32_bits(x[0]) for x in b[:3]]


def test_thread_count_determinism():
    """Results are bit-identical for 1, 3 and 8 threads (fixed chunk order)."""
    rng = np.random.default_rng(7)
    n = 400_000
    acc = rng.normal(0, 1e-3, n).astype(np.float32)
    assert len({oracle.sumsq(acc, threads=k) for k in (1, 3, 8)}) == 1
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    outs = []
    for k in (1, 3, 8):
        p = p0.copy()
        m, v, pb = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
        oracle.adamw(p, m, v, pb, acc, 0.7, grp(), 1, threads=k)
        outs.append((p, m, v, pb))
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert np.array_equal(a, b)
