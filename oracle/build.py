"""Builds liboracle.so (plain C11, FP64) in place.

-ffp-contract=off keeps every FP64 multiply and add separately rounded, so the
oracle gives the same bits on x86-64 and on aarch64.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB_PATH = os.path.join(HERE, "liboracle.so")
SOURCES = [os.path.join(HERE, "oracle.c")]
HEADERS = [os.path.join(HERE, "oracle.h"), os.path.join(ROOT, "synth", "synth.h")]


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build_cmd():
    return ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-pthread", "-o", LIB_PATH] + SOURCES + ["-lm"]


def build(force=False):
    """Compile liboracle.so if missing or older than its sources."""
    if force or _stale(LIB_PATH, SOURCES + HEADERS):
        subprocess.run(build_cmd(), check=True)
    return LIB_PATH
