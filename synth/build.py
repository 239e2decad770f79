"""Builds libsynth.so (host C) and libsynth_gpu.so (sm_103a) in place."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsynth.so")
GPU_LIB_PATH = os.path.join(HERE, "libsynth_gpu.so")
SOURCES = [os.path.join(HERE, "synth.c")]
GPU_SOURCES = [os.path.join(HERE, "synth_gpu.cu")]
HEADERS = [os.path.join(HERE, "synth.h")]


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build_cmd():
    return ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
            "-o", LIB_PATH] + SOURCES + ["-lm"]


def build_gpu_cmd():
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    nvcc = nvcc if os.path.exists(nvcc) else "nvcc"
    return [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-fmad=false",
            "-Xcompiler", "-fPIC", "-shared", "-o", GPU_LIB_PATH] + GPU_SOURCES


def build(force=False):
    """Compile libsynth.so if missing or older than its sources."""
    if force or _stale(LIB_PATH, SOURCES + HEADERS):
        subprocess.run(build_cmd(), check=True)
    return LIB_PATH


def build_gpu(force=False):
    """Compile libsynth_gpu.so if missing or older than its sources."""
    if force or _stale(GPU_LIB_PATH, GPU_SOURCES + HEADERS):
        subprocess.run(build_gpu_cmd(), check=True)
    return GPU_LIB_PATH
