"""Seeded synthetic inputs for the BF16 optimizer step (harness only).

Python front end of libsynth.so: fills host arrays with the micro-batch
gradients and initial master weights of a workload (see `workloads`), or
gathers single elements of them.  Holds none of the optimizer's arithmetic.
"""
import ctypes
import os

import numpy as np

from . import build as _build
from .workloads import Workload, Tensor, WORKLOADS, workload  # noqa: F401

SEED = 0
KIND_GRAD, KIND_MASTER, KIND_ZERO_MASK = 1, 2, 3

_lib = None


def lib():
    global _lib
    if _lib is None:
        _build.build()
        L = ctypes.CDLL(_build.LIB_PATH)
        u64, u32, i32, dbl, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.synth_stream_key.restype = u64
        L.synth_stream_key.argtypes = [u64, u32, u32, u32, u32]
        L.synth_sigma_scale.restype = dbl
        L.synth_sigma_scale.argtypes = [dbl]
        L.synth_fill_grad_bf16.argtypes = [vp, u64, u64, u64, dbl, u64, u64, i32]
        L.synth_fill_normal_f32.argtypes = [vp, u64, u64, u64, dbl, i32]
        L.synth_fill_loguniform_f32.argtypes = [vp, u64, u64, u64, i32, i32, i32]
        L.synth_gather_grad_bf16.argtypes = [vp, vp, u64, u64, dbl, u64, u64]
        L.synth_gather_normal_f32.argtypes = [vp, vp, u64, u64, dbl]
        L.synth_gather_loguniform_f32.argtypes = [vp, vp, u64, u64, i32, i32]
        for f in ("synth_fill_grad_bf16", "synth_fill_normal_f32", "synth_fill_loguniform_f32",
                  "synth_gather_grad_bf16", "synth_gather_normal_f32", "synth_gather_loguniform_f32"):
            getattr(L, f).restype = None
        _lib = L
    return _lib


def nthreads():
    return max(1, os.cpu_count() or 1)


def key(wl_id, kind, step=0, micro=0, seed=SEED):
    return lib().synth_stream_key(seed, wl_id, kind, step, micro)


def sigma_scale(sigma):
    return lib().synth_sigma_scale(sigma)


def zero_thresh(frac):
    """Forced-zero threshold on a 64-bit hash for a fraction `frac` of elements."""
    if frac <= 0:
        return 0
    return min(int(frac * 2.0 ** 64), 2 ** 64 - 1)


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def fill_grad(wl, step, micro, out, first=0, threads=None):
    """out[j] = bf16 bits of gradient element first+j of (step, micro) of workload wl."""
    assert out.dtype == np.uint16 and out.flags.c_contiguous
    lib().synth_fill_grad_bf16(_ptr(out), out.size, first, key(wl.id, KIND_GRAD, step, micro),
                               sigma_scale(wl.grad_sigma), key(wl.id, KIND_ZERO_MASK),
                               zero_thresh(wl.zero_frac), threads or nthreads())
    return out


def gather_grad(wl, step, micro, idx):
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(idx.size, np.uint16)
    lib().synth_gather_grad_bf16(_ptr(out), _ptr(idx), idx.size, key(wl.id, KIND_GRAD, step, micro),
                                 sigma_scale(wl.grad_sigma), key(wl.id, KIND_ZERO_MASK),
                                 zero_thresh(wl.zero_frac))
    return out


def _fill_tensor_master(wl, t, out, lo, hi, first, threads):
    """Fill out[lo-first : hi-first] with the initial masters of tensor t on [lo, hi)."""
    seg = out[lo - first:hi - first]
    kind = t.init[0]
    if kind == "normal":
        lib().synth_fill_normal_f32(_ptr(seg), seg.size, lo, key(wl.id, KIND_MASTER),
                                    sigma_scale(t.init[1]), threads)
    elif kind == "const":
        seg[:] = np.float32(t.init[1])
    elif kind == "loguniform":
        lib().synth_fill_loguniform_f32(_ptr(seg), seg.size, lo, key(wl.id, KIND_MASTER),
                                        t.init[1], t.init[2], threads)
    else:
        raise ValueError(kind)


def fill_master(wl, out, first=0, threads=None):
    """out[j] = initial FP32 master of element first+j of workload wl."""
    assert out.dtype == np.float32 and out.flags.c_contiguous
    end = first + out.size
    for t, off in zip(wl.tensors, wl.offsets):
        lo, hi = max(first, off), min(end, off + t.numel)
        if lo < hi:
            _fill_tensor_master(wl, t, out, lo, hi, first, threads or nthreads())
    return out


def gather_master(wl, idx):
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(idx.size, np.float32)
    tid = wl.tensor_of(idx)
    for ti in np.unique(tid):
        sel = np.nonzero(tid == ti)[0]
        t = wl.tensors[ti]
        sub = np.ascontiguousarray(idx[sel])
        tmp = np.empty(sub.size, np.float32)
        kind = t.init[0]
        if kind == "normal":
            lib().synth_gather_normal_f32(_ptr(tmp), _ptr(sub), sub.size, key(wl.id, KIND_MASTER),
                                          sigma_scale(t.init[1]))
        elif kind == "const":
            tmp[:] = np.float32(t.init[1])
        else:
            lib().synth_gather_loguniform_f32(_ptr(tmp), _ptr(sub), sub.size, key(wl.id, KIND_MASTER),
                                              t.init[1], t.init[2])
        out[sel] = tmp
    return out
