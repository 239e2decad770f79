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
    # Under a checked build of the library (BF16OPT_CHECK_FAULTS set, the build
    # named by BF16OPT_LIBRARY), any bounds or alignment violation the kernels
    # recorded during the session fails it.
    if not os.environ.get("BF16OPT_CHECK_FAULTS"):
        return
    from mixed_precision_optimizer_bf16_gb300 import bf16opt as C
    rc, bits = C.bf16opt_debug_faults()
    print(f"\nchecked build: status {rc}, fault bits {bits:#x}")
    if rc != 0 or bits != 0:
        session.exitstatus = 1
