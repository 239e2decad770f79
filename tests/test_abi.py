"""The C ABI without a GPU: build, exported symbols, struct layout, validation.

bf16opt_create validates its descriptor before touching CUDA, so every
argument error is reported the same way with or without a device.
"""
import ctypes
import os
import re
import subprocess

import pytest

from mixed_precision_optimizer_bf16_gb300 import bf16opt as C
from mixed_precision_optimizer_bf16_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bf16opt.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return C.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bf16opt_[a-z_]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(C.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True, check=True)
    syms = set(re.findall(r"\bT (bf16opt_\w+)", out.stdout))
    for name in declared_functions():
        assert name in syms, name
        assert hasattr(lib, name)


def test_struct_layout_matches_header(tmp_path):
    probe = tmp_path / "probe.c"
    probe.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "bf16opt.h"
int main(void) {
  printf("%zu %zu %zu %zu\\n", sizeof(bf16opt_desc_t), sizeof(bf16opt_tensor_t), sizeof(bf16opt_range_t), sizeof(bf16opt_group_t));
  printf("%zu %zu %zu %zu %zu %zu %zu\\n", offsetof(bf16opt_desc_t, groups), offsetof(bf16opt_desc_t, n),
         offsetof(bf16opt_desc_t, param_bf16), offsetof(bf16opt_desc_t, ranges), offsetof(bf16opt_desc_t, n_tensors),
         offsetof(bf16opt_desc_t, tensors), offsetof(bf16opt_desc_t, grad_scale));
  printf("%zu %zu\\n", offsetof(bf16opt_tensor_t, numel), offsetof(bf16opt_tensor_t, group));
  return 0;
}
""")
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(probe)], check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    sizes = [int(x) for x in lines[0].split()]
    assert sizes == [ctypes.sizeof(C.bf16opt_desc_t), ctypes.sizeof(C.bf16opt_tensor_t),
                     ctypes.sizeof(C.bf16opt_range_t), ctypes.sizeof(C.bf16opt_group_t)]
    offs = [int(x) for x in lines[1].split()]
    D = C.bf16opt_desc_t
    assert offs == [D.groups.offset, D.n.offset, D.param_bf16.offset, D.ranges.offset, D.n_tensors.offset,
                    D.tensors.offset, D.grad_scale.offset]
    T = C.bf16opt_tensor_t
    assert [int(x) for x in lines[2].split()] == [T.numel.offset, T.group.offset]


G = [dict(lr=6e-5, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.01),
     dict(lr=6e-5, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0)]
BASE = 0x7f0000000000  # fake device addresses: validation never dereferences them


def flat(n=1000, **kw):
    args = dict(master=BASE, exp_avg=BASE + 0x100000, exp_avg_sq=BASE + 0x200000, grad_accum=BASE + 0x300000,
                param_bf16=BASE + 0x400000)
    args.update({k: v for k, v in kw.items() if k in args})
    other = {k: v for k, v in kw.items() if k not in args}
    return C.flat_desc(n, args["master"], args["exp_avg"], args["exp_avg_sq"], args["grad_accum"],
                       args["param_bf16"], other.pop("groups", G), **other)


@pytest.mark.parametrize("desc,code", [
    (lambda: flat(groups=[dict(G[0], beta1=1.0)]), C.BF16OPT_ERR_INVALID_ARG),
    (lambda: flat(groups=[dict(G[0], eps=0.0)]), C.BF16OPT_ERR_INVALID_ARG),
    (lambda: flat(groups=[dict(G[0], lr=float("nan"))]), C.BF16OPT_ERR_INVALID_ARG),
    (lambda: flat(groups=[dict(G[0], weight_decay=-1.0)]), C.BF16OPT_ERR_INVALID_ARG),
    (lambda: flat(groups=G * 9), C.BF16OPT_ERR_INVALID_ARG),
    (lambda: flat(master=0), C.BF16OPT_ERR_INVALID_ARG),
    (lambda: flat(master=BASE + 2), C.BF16OPT_ERR_ALIGNMENT),
    (lambda: flat(param_bf16=BASE + 0x400001), C.BF16OPT_ERR_ALIGNMENT),
    (lambda: flat(exp_avg=BASE + 3996), C.BF16OPT_ERR_INVALID_ARG),          # overlaps master
    (lambda: flat(ranges=[(0, 500, 0), (600, 1000, 1)]), C.BF16OPT_ERR_INVALID_ARG),  # gap
    (lambda: flat(ranges=[(0, 500, 0), (400, 1000, 1)]), C.BF16OPT_ERR_INVALID_ARG),  # overlap
    (lambda: flat(ranges=[(0, 500, 0), (500, 999, 1)]), C.BF16OPT_ERR_INVALID_ARG),   # short
    (lambda: flat(ranges=[(0, 1000, 2)]), C.BF16OPT_ERR_INVALID_ARG),                # bad group
    (lambda: flat(max_grad_norm=float("inf")), C.BF16OPT_ERR_INVALID_ARG),
    (lambda: flat(grad_scale=0.0), C.BF16OPT_ERR_INVALID_ARG),
    (lambda: C.list_desc([(BASE, BASE + 4096, BASE + 8192, BASE + 12288, BASE + 16384, 1000, 0),
                          (BASE + 2000, BASE + 0x10000, BASE + 0x20000, BASE + 0x30000, BASE + 0x40000, 10, 1)], G),
     C.BF16OPT_ERR_INVALID_ARG),                                                     # tensor 1 overlaps tensor 0
    (lambda: C.list_desc([(BASE, BASE + 4096, BASE + 8192, BASE + 12288, BASE + 16385, 1000, 0)], G),
     C.BF16OPT_ERR_ALIGNMENT),
    (lambda: C.list_desc([(BASE, BASE + 4096, BASE + 8192, BASE + 12288, BASE + 16384, 1000, 5)], G),
     C.BF16OPT_ERR_INVALID_ARG),
])
def test_create_validation(lib, desc, code):
    d = desc()
    rc, h = C.bf16opt_create(d)
    assert rc == code, C.bf16opt_last_error(None)
    assert not h.value
    assert C.bf16opt_last_error(None)


def test_offload_create_validation(lib):
    """The offload variant validates its descriptor like bf16opt_create, before
    any CUDA call, and takes FLAT shards only."""
    for d in (flat(groups=[dict(G[0], beta1=1.0)]), flat(master=BASE + 2)):
        rc, h = C.bf16opt_create_offload(d)
        assert rc in (C.BF16OPT_ERR_INVALID_ARG, C.BF16OPT_ERR_ALIGNMENT) and not h.value
    lst = C.list_desc([(BASE, BASE + 4096, BASE + 8192, BASE + 12288, BASE + 16384, 1000, 0)], G)
    rc, h = C.bf16opt_create_offload(lst)
    assert rc == C.BF16OPT_ERR_INVALID_ARG and "FLAT" in C.bf16opt_last_error(None) and not h.value
    h = ctypes.c_void_p()
    assert lib.bf16opt_create_offload(None, 0, ctypes.byref(h)) == C.BF16OPT_ERR_INVALID_ARG


def test_static_norm_without_device_touches_nothing(lib):
    """Without a GPU the allocation-free norm refuses before any pointer is used
    (host arrays here stand for memory a kernel could not reach); argument
    errors are reported first, as with a device."""
    import numpy as np
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    acc, out = np.ones(1000, np.float32), np.zeros(3, np.float64)
    assert C.bf16opt_grad_norm_static(acc.ctypes.data, acc.size, 1.0, 1.0, out.ctypes.data) == \
        C.BF16OPT_ERR_UNSUPPORTED
    assert out.tolist() == [0.0, 0.0, 0.0]
    assert C.bf16opt_grad_norm_static(acc.ctypes.data, acc.size, 1.0, 1.0, out.ctypes.data + 4) == \
        C.BF16OPT_ERR_ALIGNMENT
    assert C.bf16opt_grad_norm_static(acc.ctypes.data, C.BF16OPT_STATIC_NORM_MAX_ELEMS + 1, 1.0, 1.0,
                                      out.ctypes.data) == C.BF16OPT_ERR_INVALID_ARG


def test_rank_sum_is_rank_ordered(lib):
    """bf16opt_sum_rank_sumsqs adds the per-rank values left to right in FP64
    (host only): here the order decides the result."""
    assert C.bf16opt_sum_rank_sumsqs([1.0, 1e-16, -1.0]) == (0, 0.0)
    assert C.bf16opt_sum_rank_sumsqs([1e-16, 1.0, -1.0]) == (0, 0.0)
    assert C.bf16opt_sum_rank_sumsqs([1.0, -1.0, 1e-16]) == (0, 1e-16)
    assert C.bf16opt_sum_rank_sumsqs([]) [0] == C.BF16OPT_ERR_INVALID_ARG
    assert C.bf16opt_sum_rank_sumsqs([2.5]) == (0, 2.5)
    assert C.bf16opt_set_rank_sumsqs(None, [1.0], 0)[0] == C.BF16OPT_ERR_INVALID_ARG


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.bf16opt_create(None, ctypes.byref(h)) == C.BF16OPT_ERR_INVALID_ARG
    assert C.bf16opt_accumulate(None, 0, None, C.BF16OPT_FIRST) == C.BF16OPT_ERR_INVALID_ARG
    assert C.bf16opt_grad_norm(None)[0] == C.BF16OPT_ERR_INVALID_ARG
    assert C.bf16opt_step(None) == C.BF16OPT_ERR_INVALID_ARG
    assert C.bf16opt_destroy(None) == C.BF16OPT_OK
    assert C.bf16opt_get_step(None)[0] == C.BF16OPT_ERR_INVALID_ARG
    assert C.bf16opt_set_step(None, 3) == C.BF16OPT_ERR_INVALID_ARG


def test_error_strings(lib):
    for code in (0, 1, -1, -2, -3, -4, -5, -6):
        assert C.bf16opt_error_string(code) not in ("", "unknown status")
    assert C.bf16opt_error_string(-99) == "unknown status"


def test_valid_descriptor_without_device_is_unsupported(lib):
    """With no GPU visible a valid descriptor gets ERR_UNSUPPORTED, never a crash."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    rc, h = C.bf16opt_create(flat(ranges=[(0, 400, 0), (400, 1000, 1)]))
    assert rc == C.BF16OPT_ERR_UNSUPPORTED and not h.value


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        C.load(str(tmp_path / "libbf16opt.so"))


def test_python_binding_refuses_host_tensors():
    """The binding checks what the C ABI cannot (bare pointers): state buffers
    must be contiguous CUDA tensors of the right dtype and size, and it says so
    before any CUDA call."""
    torch = pytest.importorskip("torch")
    from mixed_precision_optimizer_bf16_gb300.optimizer import BF16Optimizer
    n = 16
    flat = {k: torch.zeros(n, dtype=torch.float32) for k in ("master", "exp_avg", "exp_avg_sq", "grad_accum")}
    flat["param_bf16"] = torch.zeros(n, dtype=torch.int16)
    groups = [dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0)]
    with pytest.raises(ValueError, match="CUDA tensor"):
        BF16Optimizer(groups, flat=flat)


def test_unknown_handles_are_rejected_without_dereference(lib):
    """A pointer bf16opt_create never returned is refused by every handle call
    (the library checks a registry of live handles before touching it)."""
    fake = ctypes.c_void_p(0x10)          # never a handle; dereferencing it would crash
    E = C.BF16OPT_ERR_INVALID_ARG
    g = ctypes.c_void_p(0x1000)
    assert C.bf16opt_accumulate(fake, g.value, None, C.BF16OPT_FIRST) == E
    assert C.bf16opt_grad_norm(fake, 0, True)[0] == E
    assert C.bf16opt_grad_norm_local(fake)[0] == E
    assert C.bf16opt_set_global_sumsq(fake, 1.0) == E
    assert C.bf16opt_step(fake) == E
    assert C.bf16opt_get_step(fake)[0] == E
    assert C.bf16opt_set_step(fake, 3) == E
    assert C.bf16opt_set_skip_nonfinite(fake, True) == E
    assert C.bf16opt_set_lr_schedule(fake, C.lr_schedule(10, 100, 0.1)) == E
    assert C.bf16opt_step_path(fake) == (E, C.BF16OPT_PATH_NONE)
    assert C.bf16opt_destroy(fake) == E
    assert "not a live" in C.bf16opt_last_error(fake)


def test_pipeline_timeouts_without_device(lib):
    """The pipeline's timeout count needs a device: without one the call says
    so instead of touching CUDA state; a NULL output is an argument error."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    assert C.bf16opt_pipeline_timeouts() == (C.BF16OPT_ERR_UNSUPPORTED, 0)
    assert lib.bf16opt_pipeline_timeouts(None) == C.BF16OPT_ERR_INVALID_ARG


def test_abi_version_matches_header_and_binding(lib):
    """The library, the header and the Python binding agree on the ABI version."""
    src = open(HEADER).read()
    m = re.search(r"#define BF16OPT_ABI_VERSION (\d+)", src)
    assert m and int(m.group(1)) == C.ABI_VERSION == lib.bf16opt_abi_version()
