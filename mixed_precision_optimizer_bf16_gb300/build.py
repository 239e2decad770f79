"""Builds libbf16opt.so (the C-ABI library and its sm_103a kernels) in place."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB_PATH = os.path.join(HERE, "libbf16opt.so")
SOURCES = [os.path.join(HERE, "csrc", "bf16opt.cu")]
DEPS = SOURCES + [os.path.join(HERE, "csrc", "kernels.cuh"), os.path.join(HERE, "csrc", "host_adam.h"),
                  os.path.join(ROOT, "include", "bf16opt.h")]

# -ffp-contract=off: host code rounds every product on its own (the offloaded
# step's host update repeats the device kernel's operations exactly)
PROBE_LIB_PATH = os.path.join(HERE, "libhbmprobe.so")
PROBE_SOURCES = [os.path.join(HERE, "csrc", "hbm_probe.cu")]
PROBE_DEPS = PROBE_SOURCES + [os.path.join(ROOT, "include", "hbm_probe.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off", "-shared"]


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build_cmd(extra=(), out=None):
    return [nvcc()] + NVCC_FLAGS + list(extra) + ["-I", os.path.join(ROOT, "include"), "-o", out or LIB_PATH] + SOURCES


def build_probe_cmd():
    return [nvcc()] + NVCC_FLAGS + ["-I", os.path.join(ROOT, "include"), "-o", PROBE_LIB_PATH] + PROBE_SOURCES


def build_probe(force=False):
    """Compile libhbmprobe.so (the HBM bandwidth probe) if missing or stale."""
    if force or _stale(PROBE_LIB_PATH, PROBE_DEPS):
        subprocess.run(build_probe_cmd(), check=True)
    return PROBE_LIB_PATH


def build_checked(out):
    """Compile the checked variant (-DBF16K_CHECKS: kernels test chunk ranges
    and vector alignment and record violations instead of accessing) to `out`."""
    subprocess.run(build_cmd(["-DBF16K_CHECKS=1"], out), check=True)
    return out


def build(force=False, extra=()):
    """Compile libbf16opt.so for sm_103a if missing or older than its sources."""
    if force or _stale(LIB_PATH, DEPS):
        subprocess.run(build_cmd(extra), check=True)
    return LIB_PATH
