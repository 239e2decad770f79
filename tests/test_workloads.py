"""The workload tables against the numbers the pages print (tests/golden/pages_numbers.txt)."""
import os

import numpy as np

from synth import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.txt")


def golden():
    out = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = float(v)
    return out


def test_hyperparameters_from_pages():
    g = golden()
    for wl in workloads.WORKLOADS.values():
        assert wl.groups[0]["lr"] == g["lr"]
        assert wl.groups[0]["weight_decay"] == g["weight_decay"]
        assert wl.groups[1]["weight_decay"] == 0.0
        assert wl.max_norm == g["clip_grad"]
    assert workloads.workload(2).gas == g["gas_scaled"]
    assert workloads.workload(3).gas == g["gas_bloom176"]


def test_scaled_bloom_shapes():
    """hidden 2048, 24 layers, vocab 250880, tied embeddings: 293 tensors and
    1,722,408,960 parameters (the "1.72B" of the workload), 647,168 of them in
    LayerNorm/bias tensors."""
    g = golden()
    wl = workloads.workload(2)
    h, L, V = int(g["hidden_scaled"]), int(g["layers_scaled"]), int(g["vocab"])
    per_layer = 12 * h * h + 13 * h
    assert wl.n == V * h + 4 * h + L * per_layer == 1_722_408_960
    assert len(wl.tensors) == 293
    assert sum(t.numel for t in wl.tensors if not t.decay) == 647_168
    r = wl.ranges()
    assert r[0][0] == 0 and r[-1][1] == wl.n
    assert all(a[1] == b[0] for a, b in zip(r, r[1:]))


def test_bloom176_tp4_slice_shapes():
    """Six BLOOM-176B layers (hidden 14336) cut 4 ways: 72 tensors, 3,700,064,256 elements."""
    g = golden()
    h, tp = int(g["hidden_bloom176"]), int(g["tp_degree"])
    wl = workloads.workload(4)
    assert wl.mode == "list" and len(wl.tensors) == 72
    per_layer = (3 * h // tp) * h + h * (h // tp) + 2 * (4 * h // tp) * h + 8 * h
    assert wl.n == 6 * per_layer == 3_700_064_256
    assert sum(t.numel for t in wl.tensors if not t.decay) == 688_128


def test_other_workloads():
    assert workloads.workload(1).n == 1 << 20
    assert workloads.workload(3).n == 1_830_000_000
    w5 = workloads.workload(5)
    assert w5.n == (1 << 27) + 13 and w5.misalign == 2 and w5.zero_frac == 0.01


def test_bytes_model():
    """Algorithmic bytes per element: 6 (first micro-batch) + 10 per later one + 30 (fused step)."""
    wl = workloads.workload(2)
    assert wl.bytes_per_step() == wl.n * 66
    assert workloads.workload(3).bytes_per_step() == workloads.workload(3).n * (6 + 310 + 30)
    np.testing.assert_equal(wl.tensor_of([0, 513_802_239, 513_802_240]), [0, 0, 1])


def test_resident_pattern_respects_the_pending_limit():
    """resident_pattern never leaves more than 8 micro-batches pending, defers
    everything for GAS <= 8, and ends every pattern deferred."""
    from mixed_precision_optimizer_bf16_gb300.optimizer import resident_pattern
    for gas in range(1, 70):
        pat = resident_pattern(gas)
        assert len(pat) == gas and pat[-1]
        run = worst = 0
        for d in pat:
            run = run + 1 if d else 0
            worst = max(worst, run)
        assert worst <= 8
        assert all(pat) == (gas <= 8)
