"""The library used from plain C, through include/bf16opt.h alone.

tests/c_abi/step_parity.c runs two optimizer steps through the C ABI with
device memory from the CUDA runtime and checks them against the C oracle on
the same seeded inputs (see its header).  Compiling and linking it needs no
GPU; running it does.
"""
import os
import subprocess

import pytest

from mixed_precision_optimizer_bf16_gb300 import build as B
from oracle import build as OB

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
SRC = os.path.join(ROOT, "tests", "c_abi", "step_parity.c")


def _compile(out_dir):
    B.build()
    OB.build()
    exe = os.path.join(str(out_dir), "step_parity")
    libdirs = [os.path.dirname(B.LIB_PATH), os.path.dirname(OB.LIB_PATH), os.path.join(CUDA, "lib64")]
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-o", exe, SRC,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "oracle"), "-I", os.path.join(ROOT, "synth"),
           "-I", os.path.join(CUDA, "include")]
    for d in libdirs:
        cmd += ["-L", d]
    cmd += ["-lbf16opt", "-loracle", "-lcudart", "-lm", "-Wl,-rpath," + ":".join(libdirs)]
    subprocess.run(cmd, check=True)
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(_compile(tmp_path))


@pytest.mark.gpu
def test_c_program_matches_oracle(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout, r.stderr)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok" in r.stdout


@pytest.mark.parametrize("lang, std", [("c", "c99"), ("c++", "c++11"), ("c++", "c++17")])
def test_header_compiles_standalone(tmp_path, lang, std):
    """include/bf16opt.h on its own: plain C99 (pedantic) and C++, warnings as errors."""
    src = tmp_path / ("use.c" if lang == "c" else "use.cpp")
    src.write_text('#include "bf16opt.h"\n'
                   "int probe(void) { bf16opt_desc_t d; (void)d; return BF16OPT_ABI_VERSION + BF16OPT_MAX_GROUPS; }\n")
    cc = "gcc" if lang == "c" else "g++"
    subprocess.run([cc, f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror", "-c", str(src),
                    "-I", os.path.join(ROOT, "include"), "-o", str(tmp_path / "use.o")], check=True)
