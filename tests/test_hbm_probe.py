"""The HBM bandwidth probe (include/hbm_probe.h, libhbmprobe.so): exports,
argument checks without a GPU, and on a GPU that the copy kernel copies and
every mix reports a plausible bandwidth."""
import os
import re
import subprocess

import pytest

from mixed_precision_optimizer_bf16_gb300 import build as B
from mixed_precision_optimizer_bf16_gb300 import hbm_probe as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build_probe()
    return P.load()


def test_header_and_library_exports(lib):
    src = open(os.path.join(ROOT, "include", "hbm_probe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    declared = sorted(set(re.findall(r"\b(hbm_probe_[a-z_]+)\s*\(", src)))
    assert declared == sorted(P.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", B.PROBE_LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    for name in declared:
        assert re.search(r"\bT " + name + r"\b", out), name


def test_arguments_are_checked_before_any_device_work(lib):
    fake = [0x7f0000000000 + 4096 * i for i in range(6)]
    assert P.hbm_probe_run(P.HBM_PROBE_COPY, fake, 4095)[0] == -1          # not whole chunks
    assert P.hbm_probe_run(9, fake, 4096)[0] == -1                          # unknown kind
    assert P.hbm_probe_run(P.HBM_PROBE_COPY, [fake[0] + 8, fake[1]], 4096)[0] == -1   # misaligned
    assert P.hbm_probe_run(P.HBM_PROBE_STEP_MIX, fake[:5] + [0], 4096)[0] == -1       # NULL buffer
    assert P.hbm_probe_run(P.HBM_PROBE_COPY, fake[:2], 4096, reps=0)[0] == -1


@pytest.mark.gpu
def test_probe_on_the_gpu(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    n = 1 << 24                                    # 256 MiB per buffer: beyond L2
    a = torch.randn(n * 4, device="cuda")
    b = torch.zeros(n * 4, device="cuda")
    rc, ms, nbytes = P.hbm_probe_run(P.HBM_PROBE_COPY, [a.data_ptr(), b.data_ptr()], n)
    torch.cuda.synchronize()
    assert rc == 0 and ms > 0 and nbytes == 32 * n
    assert torch.equal(a, b)                       # every chunk copied exactly once
    # the bulk-copy kinds move every tile exactly once: one launch of the
    # accumulate mix adds g to acc once per element, one launch of the step
    # mix adds a to p once per element and writes p's high halves as bf16
    q = 1 << 22
    g = torch.randint(-2**14, 2**14, (q * 4,), dtype=torch.int16, device="cuda")   # finite bf16 values
    acc = torch.randn(q * 4, device="cuda")
    want = acc + (g.to(torch.int32) << 16).view(torch.float32)
    rc, ms, nbytes = P.hbm_probe_run(P.HBM_PROBE_BULK_ACC_MIX, [g.data_ptr(), acc.data_ptr()], q, warmup=0, reps=1)
    torch.cuda.synchronize()
    assert rc == 0 and nbytes == 40 * q
    assert torch.equal(acc.view(torch.int32), want.view(torch.int32))
    bufs = [torch.randn(q * 4, device="cuda"), g, torch.randn(q * 4, device="cuda"), torch.randn(q * 4, device="cuda"),
            torch.randn(q * 4, device="cuda"), torch.zeros(q * 4, dtype=torch.int16, device="cuda")]
    p_want = bufs[2] + bufs[0]
    rc, ms, nbytes = P.hbm_probe_run(P.HBM_PROBE_BULK_STEP_MIX, [t.data_ptr() for t in bufs], q, warmup=0, reps=1)
    torch.cuda.synchronize()
    assert rc == 0 and nbytes == 128 * q
    assert torch.equal(bufs[2].view(torch.int32), p_want.view(torch.int32))
    assert torch.equal(bufs[5], (p_want.view(torch.int32) >> 16).to(torch.int16))
    got = P.measure(vectors=n, quads=n // 2)
    for k in ("copy_gbs", "write_gbs", "read_gbs", "step_mix_gbs", "first_mix_gbs", "acc_mix_gbs",
              "step_mix_bulk_gbs", "acc_mix_bulk_gbs"):
        assert 500.0 < got[k] < 20000.0, (k, got)
