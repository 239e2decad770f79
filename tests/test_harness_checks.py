"""The parity checks themselves: harness.compare must catch a planted error
just beyond its tolerance in any state, and let one well inside it pass --
otherwise the GPU parity tests would prove nothing.  CPU only: the "GPU"
result is the oracle's own result with the error planted."""
import numpy as np
import pytest

import harness
from harness import REL, compare, oracle_dense
from synth import workloads


@pytest.fixture(scope="module")
def ref_run():
    wl = workloads.custom(901, [5000, 777], decay=[True, False], gas=2, steps=2, grad_sigma=0.2)
    ref, scales = oracle_dense(wl, wl.steps)
    return wl, ref, scales


def _copy(ref):
    return {k: (np.array(v, copy=True) if isinstance(v, np.ndarray) else v) for k, v in ref.items()}


def test_identical_result_passes(ref_run):
    wl, ref, scales = ref_run
    compare(_copy(ref), ref, scales, wl)


@pytest.mark.parametrize("name, scale_key", [("m", "M"), ("v", None), ("p", "A")])
@pytest.mark.parametrize("factor, ok", [(0.4, True), (3.0, False)])
def test_planted_state_errors(ref_run, name, scale_key, factor, ok):
    wl, ref, scales = ref_run
    got = _copy(ref)
    i = 1234
    y = float(ref[name][i])
    s = scales[scale_key][i] if scale_key else abs(y)
    lim = max(REL * max(abs(y), s), wl.steps * harness.SUBNORMAL_UNIT)
    got[name][i] = np.float32(y + factor * lim)
    if name == "p":   # keep the bf16 copy consistent with the planted master
        import oracle
        got["p_bf16"][i] = oracle.f32_to_bf16(got["p"][i:i + 1])[0]
    if ok:
        compare(got, ref, scales, wl)
    else:
        with pytest.raises(AssertionError):
            compare(got, ref, scales, wl)


def test_bf16_not_the_cast_of_the_master_is_caught(ref_run):
    wl, ref, scales = ref_run
    got = _copy(ref)
    got["p_bf16"][42] ^= 1                       # one ulp off the RNE cast of the master
    with pytest.raises(AssertionError):
        compare(got, ref, scales, wl)


def test_accumulator_bit_flip_is_caught(ref_run):
    wl, ref, scales = ref_run
    got = _copy(ref)
    got["acc"][7] = np.nextafter(got["acc"][7], np.float32(np.inf))
    with pytest.raises(AssertionError):
        compare(got, ref, scales, wl)


def test_bf16_half_ulp():
    got = harness._bf16_half_ulp(np.array([1.0, 1.5, 2.0, -3.0, 0.0, 2.0 ** -130, 2.0 ** -126], np.float32))
    # bf16 keeps 8 significant bits: the unit at 1.0 is 2^-7, below 2^-126 it is 2^-133
    assert got.tolist() == [2.0 ** -8, 2.0 ** -8, 2.0 ** -7, 2.0 ** -7, 2.0 ** -134, 2.0 ** -134, 2.0 ** -134]


def test_bf16_several_units_off_pass_only_where_the_master_cancels(ref_run):
    """A master that cancels far below its operand scale A has an FP32
    tolerance (1e-6 A) wider than a bf16 unit: its bf16 may then lie several
    units from the oracle's, and compare() counts it."""
    import oracle
    wl, ref, scales = ref_run
    got, sc = _copy(ref), {k: np.array(v, copy=True) for k, v in scales.items()}
    i = 99
    ref2 = _copy(ref)
    ref2["p"][i] = np.float32(1e-9)
    ref2["p_bf16"][i] = oracle.f32_to_bf16(ref2["p"][i:i + 1])[0]
    sc["A"][i] = 1.0                                 # operand scale: tolerance 1e-6
    got["p"][i] = np.float32(1e-9 + 5e-7)
    got["p_bf16"][i] = oracle.f32_to_bf16(got["p"][i:i + 1])[0]
    st = compare(got, ref2, sc, wl)
    assert st["bf16_diffs_over_1ulp"] == 1 and st["bf16_max_ulp_diff"] > 1


def _slices(n, step):
    return [(lo, min(n, lo + step)) for lo in range(0, n, step)]


def test_streamed_oracle_slices_equal_the_dense_run():
    """The full-size dense comparison runs the oracle one slice at a time with
    the global clip coefficients streamed from the counters: the slices, put
    together, must be the whole-shard run bit for bit (states, operand scales,
    and the accumulator after any number of micro-batches)."""
    import oracle
    import synth
    wl = workloads.custom(902, [40_001, 333, 12_000], decay=[True, False, True], gas=3, steps=2, grad_sigma=0.3,
                          zero_frac=0.05)
    ref, scales = oracle_dense(wl, wl.steps)
    st = oracle.stream(wl.id, wl.gas, synth.sigma_scale(wl.grad_sigma), synth.zero_thresh(wl.zero_frac))
    sums = [oracle.stream_sumsq(st, s, wl.n) for s in range(wl.steps)]
    assert sums == ref["sumsq"]
    clips = [oracle.clip_coef(S, wl.max_norm) for S in sums]
    parts = [harness._oracle_slice(wl, lo, hi, wl.steps, clips, {1, 2}, 2) for lo, hi in _slices(wl.n, 9_999)]
    for k in ("p", "m", "v", "p_bf16", "acc"):
        assert np.concatenate([p[0][k] for p in parts]).tobytes() == ref[k].tobytes(), k
    for k in ("M", "A"):
        assert np.concatenate([p[1][k] for p in parts]).tobytes() == scales[k].tobytes(), k
    for j in (1, 2):
        acc = np.empty(wl.n, np.float32)
        for k in range(j):
            oracle.accumulate(acc, synth.fill_grad(wl, wl.steps - 1, k, np.empty(wl.n, np.uint16)), first=k == 0)
        assert np.concatenate([p[2][j] for p in parts]).tobytes() == acc.tobytes()


class _FakeShard:
    """Stands in for a GpuShard: its "device" states are the oracle's dense run,
    optionally with one planted error."""

    def __init__(self, states, pattern):
        self.s, self.pattern = states, pattern

    acc_folded = harness.GpuShard.acc_folded

    def slice_states(self, lo, hi):
        return {k: np.array(v[lo:hi], copy=True) for k, v in self.s.items() if isinstance(v, np.ndarray)}


def test_dense_streamed_parity_machinery():
    wl = workloads.custom(903, [30_001, 777], decay=[True, False], gas=2, steps=2, grad_sigma=0.2)
    ref, _ = oracle_dense(wl, wl.steps)
    good = {"stored": _FakeShard(ref, [False, False])}
    stats, sums = harness.dense_streamed_parity(wl, good, wl.steps, slice_elems=7_000, workers=3)
    assert sums == ref["sumsq"] and stats["stored"]["elements"] == wl.n
    bad = {k: np.array(v, copy=True) for k, v in ref.items() if isinstance(v, np.ndarray)}
    bad["acc"][25_000] = np.nextafter(bad["acc"][25_000], np.float32(1))
    with pytest.raises(AssertionError):
        harness.dense_streamed_parity(wl, {"stored": _FakeShard(bad, [False, False])}, wl.steps,
                                      slice_elems=7_000, workers=3)
