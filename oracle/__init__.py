"""CPU oracle of the BF16Optimizer step -- TEST INFRASTRUCTURE ONLY.

Only tests/, the package smoke check and bench.py's CPU-baseline/reference leg
may import this module.  The product path never does, and it shares no code
with the CUDA library.  liboracle.so (oracle.c) evaluates the plain definition
in FP64 and rounds at the storage points; this file only marshals numpy arrays
and runs the steps in the method's order:

  for each step: accumulate micro-batches 0..GAS-1 in order (FP32 storage),
  global sum of squares, clip coefficient, AdamW per group, bf16 cast.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


class Group(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double)]


class Stream(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("workload", ctypes.c_uint32), ("gas", ctypes.c_uint32),
                ("grad_sigma_scale", ctypes.c_double), ("zero_thresh", ctypes.c_uint64),
                ("grad_scale", ctypes.c_float), ("pad", ctypes.c_uint32)]


def lib():
    global _lib
    if _lib is None:
        _build.build()
        L = ctypes.CDLL(_build.LIB_PATH)
        vp, u64, i32, i64, dbl, flt = (ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int64,
                                       ctypes.c_double, ctypes.c_float)
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_f32_to_bf16.argtypes = [flt]
        L.orc_bf16_to_f32.restype = flt
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f32_to_bf16_array.argtypes = [vp, vp, u64, i32]
        L.orc_accumulate.argtypes = [vp, vp, u64, i32, i32]
        L.orc_sumsq.restype = dbl
        L.orc_sumsq.argtypes = [vp, u64, flt, i32]
        L.orc_clip_coef.restype = dbl
        L.orc_clip_coef.argtypes = [dbl, dbl]
        L.orc_adamw.argtypes = [vp, vp, vp, vp, vp, u64, flt, dbl, ctypes.POINTER(Group), i64, i32]
        L.orc_stream_sumsq.restype = dbl
        L.orc_stream_sumsq.argtypes = [ctypes.POINTER(Stream), ctypes.c_uint32, u64, i32]
        L.orc_sample_run.argtypes = [ctypes.POINTER(Stream), vp, u64, vp, ctypes.POINTER(Group), vp,
                                     ctypes.c_uint32, vp, i64, vp, vp, vp, vp, vp]
        L.orc_lr_at.restype = dbl
        L.orc_lr_at.argtypes = [dbl, dbl, i64, i64, i64]
        for f in ("orc_f32_to_bf16_array", "orc_accumulate", "orc_adamw", "orc_sample_run"):
            getattr(L, f).restype = None
        _lib = L
    return _lib


def nthreads():
    return max(1, os.cpu_count() or 1)


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


def group(lr, beta1, beta2, eps, weight_decay):
    return Group(lr, beta1, beta2, eps, weight_decay)


def f32_to_bf16(x, threads=None):
    x = _f32(x)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16_array(_p(x), _p(out), x.size, threads or nthreads())
    return out


def bf16_to_f32(h):
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def accumulate(acc, g, first, threads=None):
    assert acc.dtype == np.float32 and g.dtype == np.uint16 and acc.size == g.size
    lib().orc_accumulate(_p(acc), _p(g), acc.size, int(bool(first)), threads or nthreads())
    return acc


def sumsq(acc, grad_scale=1.0, threads=None):
    acc = _f32(acc)
    return lib().orc_sumsq(_p(acc), acc.size, grad_scale, threads or nthreads())


def clip_coef(s, max_norm):
    return lib().orc_clip_coef(s, max_norm)


def adamw(p, m, v, pbf, acc, clip, grp, t, grad_scale=1.0, threads=None):
    for a in (p, m, v, acc):
        assert a.dtype == np.float32 and a.flags.c_contiguous
    assert pbf.dtype == np.uint16
    lib().orc_adamw(_p(p), _p(m), _p(v), _p(pbf), _p(acc), p.size, grad_scale, clip, ctypes.byref(grp), t,
                    threads or nthreads())


def stream(wl_id, gas, sigma_scale, zero_thresh=0, grad_scale=1.0, seed=0):
    return Stream(seed, wl_id, gas, sigma_scale, zero_thresh, grad_scale, 0)


def stream_sumsq(st, step, n, threads=None):
    return lib().orc_stream_sumsq(ctypes.byref(st), step, n, threads or nthreads())


def sample_run(st, idx, p0, groups, group_of, clips, t0=0):
    """Whole steps on sampled elements; returns (p, m, v, p_bf16, last acc)."""
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    k = idx.size
    p0 = _f32(p0)
    gof = np.ascontiguousarray(group_of, dtype=np.uint32)
    clips = np.ascontiguousarray(clips, dtype=np.float64)
    garr = (Group * len(groups))(*groups)
    p, m, v = (np.empty(k, np.float32) for _ in range(3))
    pb = np.empty(k, np.uint16)
    acc = np.empty(k, np.float32)
    lib().orc_sample_run(ctypes.byref(st), _p(idx), k, _p(p0), garr, _p(gof), clips.size, _p(clips), t0,
                         _p(p), _p(m), _p(v), _p(pb), _p(acc))
    return p, m, v, pb, acc


def run_dense(p, grads_fn, ranges, groups, steps, gas, max_norm, grad_scale=1.0, t0=0, m=None, v=None,
              threads=None):
    """Full oracle run over materialised host arrays.

    p: FP32 masters (updated in place); grads_fn(step, micro) -> uint16 array of
    the whole buffer, step counted from 0 (step index t0 + s has step number t0 + s + 1); ranges: [(begin, end, group index)] tiling [0, n);
    groups: list of Group.  Returns dict with p, m, v, p_bf16, acc (last step)
    and per-step sumsq / clip lists.
    """
    n = p.size
    m = np.zeros(n, np.float32) if m is None else m
    v = np.zeros(n, np.float32) if v is None else v
    pbf = f32_to_bf16(p)
    acc = np.zeros(n, np.float32)
    sums, clips = [], []
    for s in range(steps):
        for k in range(gas):
            accumulate(acc, grads_fn(t0 + s, k), first=(k == 0), threads=threads)
        S = sumsq(acc, grad_scale, threads)
        c = clip_coef(S, max_norm)
        sums.append(S)
        clips.append(c)
        for b, e, gi in ranges:
            adamw(p[b:e], m[b:e], v[b:e], pbf[b:e], acc[b:e], c, groups[gi], t0 + s + 1, grad_scale, threads)
    return dict(p=p, m=m, v=v, p_bf16=pbf, acc=acc, sumsq=sums, clip=clips)


def lr_at(lr, min_lr, warmup, decay, t):
    """Warmup + cosine learning rate at step number t >= 1."""
    return lib().orc_lr_at(lr, min_lr, warmup, decay, t)
