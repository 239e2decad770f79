"""Device-side fills of a workload's seeded inputs (libsynth_gpu.so; harness only).

Bit-identical to the host generator in synth/__init__.py: gradients and
masters for element i depend only on (workload, kind, step, micro-batch, i).
"""
import ctypes

import torch

from . import KIND_GRAD, KIND_MASTER, KIND_ZERO_MASK, build as _build, key, sigma_scale, zero_thresh

_lib = None


def lib():
    global _lib
    if _lib is None:
        _build.build_gpu()
        L = ctypes.CDLL(_build.GPU_LIB_PATH)
        u64, dbl, vp, i32 = ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        L.synth_gpu_fill_grad_bf16.argtypes = [vp, u64, u64, u64, dbl, u64, u64, vp]
        L.synth_gpu_fill_normal_f32.argtypes = [vp, u64, u64, u64, dbl, vp]
        L.synth_gpu_fill_loguniform_f32.argtypes = [vp, u64, u64, u64, i32, i32, vp]
        for f in ("synth_gpu_fill_grad_bf16", "synth_gpu_fill_normal_f32", "synth_gpu_fill_loguniform_f32"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _stream(stream):
    return ctypes.c_void_p((stream or torch.cuda.current_stream()).cuda_stream)


def fill_grad(wl, step, micro, dst, first=0, stream=None):
    """dst (int16/bf16-bits device tensor) <- gradient elements [first, first+numel)."""
    assert dst.is_cuda and dst.element_size() == 2 and dst.is_contiguous()
    rc = lib().synth_gpu_fill_grad_bf16(ctypes.c_void_p(dst.data_ptr()), dst.numel(), first,
                                        key(wl.id, KIND_GRAD, step, micro), sigma_scale(wl.grad_sigma),
                                        key(wl.id, KIND_ZERO_MASK), zero_thresh(wl.zero_frac), _stream(stream))
    if rc:
        raise RuntimeError("synth_gpu_fill_grad_bf16 failed")
    return dst


def fill_master(wl, dst, first=0, stream=None):
    """dst (float32 device tensor) <- initial masters of elements [first, first+numel)."""
    assert dst.is_cuda and dst.dtype == torch.float32 and dst.is_contiguous()
    end = first + dst.numel()
    for t, off in zip(wl.tensors, wl.offsets):
        lo, hi = max(first, off), min(end, off + t.numel)
        if lo >= hi:
            continue
        seg = dst[lo - first:hi - first]
        kind = t.init[0]
        if kind == "normal":
            rc = lib().synth_gpu_fill_normal_f32(ctypes.c_void_p(seg.data_ptr()), seg.numel(), lo,
                                                 key(wl.id, KIND_MASTER), sigma_scale(t.init[1]), _stream(stream))
        elif kind == "const":
            seg.fill_(float(t.init[1]))
            rc = 0
        else:
            rc = lib().synth_gpu_fill_loguniform_f32(ctypes.c_void_p(seg.data_ptr()), seg.numel(), lo,
                                                     key(wl.id, KIND_MASTER), t.init[1], t.init[2], _stream(stream))
        if rc:
            raise RuntimeError("synth_gpu fill failed")
    return dst
