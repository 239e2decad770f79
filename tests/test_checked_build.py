"""The GPU parity suite under the checked build of the library.

The checked build (-DBF16K_CHECKS) makes every kernel test, before each
chunk's accesses, that the chunk lies inside its segment, that its vector body
stays inside the chunk and that every vector pointer is aligned, recording a
violation in a device word instead of making the access.  It stands in for a
memory checker: this test reruns the GPU parity tests, the allocation-free norm
and the offload tests against that build and fails if any fault bit was set
(the every-element full-size comparisons stay with the release build: they
cover no code the smaller shards miss).
The release build compiles the tests away.
"""
import os
import subprocess
import sys

import pytest

from mixed_precision_optimizer_bf16_gb300 import bf16opt as C
from mixed_precision_optimizer_bf16_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_release_build_has_no_fault_word():
    B.build()
    rc, bits = C.bf16opt_debug_faults()
    assert rc == C.BF16OPT_ERR_UNSUPPORTED and bits == 0


@pytest.mark.gpu
def test_parity_suite_under_checked_build(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = B.build_checked(str(tmp_path / "libbf16opt_checked.so"))
    env = dict(os.environ, BF16OPT_LIBRARY=lib, BF16OPT_CHECK_FAULTS="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_parity_gpu.py"), os.path.join(ROOT, "tests", "test_offload_gpu.py"),
           os.path.join(ROOT, "tests", "test_zz_no_alloc.py")]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-15:])
    print(tail)
    assert r.returncode == 0, tail
    assert "fault bits 0x0" in r.stdout, tail
