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
