import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libbf16opt.so")
    config.addinivalue_line("markers", "slow: long-running check")


def pytest_collection_modifyitems(config, items):
    # Keep the no-allocation entry-point file last even if names change.
    items.sort(key=lambda it: 1 if os.path.basename(str(it.fspath)).startswith("test_zz_") else 0)


def pytest_sessionfinish(session, exitstatus):
    # Every bounded wait of the fused step's copy pipeline completed: a wait that
    # gave up during the session fails it (checked only where a GPU ran the tests).
    from mixed_precision_optimizer_bf16_gb300 import bf16opt as C
    if C._lib is not None and "torch" in sys.modules and sys.modules["torch"].cuda.is_available():
        rc, n = C.bf16opt_pipeline_timeouts()
        print(f"\nstep pipeline: status {rc}, timed-out waits {n}")
        if rc != 0 or n != 0:
            session.exitstatus = 1
    # Under a checked build of the library (BF16OPT_CHECK_FAULTS set, the build
    # named by BF16OPT_LIBRARY), any bounds or alignment violation the kernels
    # recorded during the session fails it.
    if not os.environ.get("BF16OPT_CHECK_FAULTS"):
        return
    rc, bits = C.bf16opt_debug_faults()
    print(f"\nchecked build: status {rc}, fault bits {bits:#x}")
    if rc != 0 or bits != 0:
        session.exitstatus = 1
