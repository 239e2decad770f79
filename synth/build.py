"""Builds libsynth.so (host C, seeded input generators) in place."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsynth.so")
SOURCES = [os.path.join(HERE, "synth.c")]
HEADERS = [os.path.join(HERE, "synth.h")]


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build_cmd():
    return ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
            "-o", LIB_PATH] + SOURCES + ["-lm"]


def build(force=False):
    """Compile libsynth.so if missing or older than its sources."""
    if force or _stale(LIB_PATH, SOURCES + HEADERS):
        subprocess.run(build_cmd(), check=True)
    return LIB_PATH
