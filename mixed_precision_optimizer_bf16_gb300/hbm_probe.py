"""Python binding of libhbmprobe.so (include/hbm_probe.h): argument marshalling
for the HBM bandwidth probe, and `measure`, which allocates the buffers with
torch and returns the bandwidth each traffic mix reaches on the current GPU."""
import ctypes
import os

from . import build as _build

HBM_PROBE_COPY, HBM_PROBE_WRITE, HBM_PROBE_READ, HBM_PROBE_STEP_MIX = 0, 1, 2, 3
HBM_PROBE_FIRST_MIX, HBM_PROBE_ACC_MIX = 4, 5
HBM_PROBE_BULK_STEP_MIX, HBM_PROBE_BULK_ACC_MIX = 6, 7
EXPORTS = ("hbm_probe_run", "hbm_probe_sink_bytes")

_lib = None


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(_build.PROBE_LIB_PATH):
            raise RuntimeError(f"libhbmprobe.so is not built ({_build.PROBE_LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(_build.PROBE_LIB_PATH)
        L.hbm_probe_run.restype = ctypes.c_int
        L.hbm_probe_run.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.c_uint64, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_float),
                                    ctypes.POINTER(ctypes.c_double)]
        L.hbm_probe_sink_bytes.restype = ctypes.c_int
        L.hbm_probe_sink_bytes.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
        _lib = L
    return _lib


def hbm_probe_run(kind, ptrs, n, warmup=3, reps=10, stream=0):
    """Returns (status, ms per launch, bytes per launch)."""
    arr = (ctypes.c_void_p * len(ptrs))(*[ctypes.c_void_p(int(p)) for p in ptrs])
    ms, b = ctypes.c_float(0.0), ctypes.c_double(0.0)
    rc = load().hbm_probe_run(kind, arr, n, warmup, reps, ctypes.c_void_p(int(stream)) if stream else None,
                              ctypes.byref(ms), ctypes.byref(b))
    return rc, ms.value, b.value


def hbm_probe_sink_bytes():
    b = ctypes.c_uint64(0)
    rc = load().hbm_probe_sink_bytes(ctypes.byref(b))
    return rc, b.value


def measure(vectors=1 << 28, quads=1 << 28, device="cuda", reps=10):
    """GB/s of each traffic mix on `device`: copy (1:1) and write-only and
    read-only over buffers of `vectors` 16-byte vectors; the fused step's
    18:14 mix and the accumulate passes' 2:4 (first) and 6:4 (later) mixes over
    `quads` 4-element quads, with vector loads, and the step's and a later
    accumulate's mixes through bulk copies (`*_bulk_gbs`).  Allocates and frees
    the buffers."""
    import torch
    out = {}
    stream = torch.cuda.current_stream(device).cuda_stream
    a = torch.empty(vectors * 4, dtype=torch.float32, device=device)
    b = torch.empty(vectors * 4, dtype=torch.float32, device=device)
    a.fill_(1.0)
    rc, sink = hbm_probe_sink_bytes()
    if rc:
        raise RuntimeError(f"hbm_probe_sink_bytes failed ({rc})")
    s = torch.zeros(max(1, sink // 4), dtype=torch.int32, device=device)
    for name, kind, ptrs in (("copy", HBM_PROBE_COPY, [a.data_ptr(), b.data_ptr()]),
                             ("write", HBM_PROBE_WRITE, [b.data_ptr()]),
                             ("read", HBM_PROBE_READ, [a.data_ptr(), s.data_ptr()])):
        rc, ms, nbytes = hbm_probe_run(kind, ptrs, vectors, 3, reps, stream)
        if rc:
            raise RuntimeError(f"hbm_probe_run({name}) failed ({rc})")
        out[name + "_gbs"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
    del a, b, s
    bufs = [torch.zeros(quads * k, dtype=dt, device=device) for k, dt in
            ((4, torch.float32), (4, torch.int16), (4, torch.float32), (4, torch.float32), (4, torch.float32),
             (4, torch.int16))]
    for name, kind in (("step_mix_gbs", HBM_PROBE_STEP_MIX), ("step_mix_bulk_gbs", HBM_PROBE_BULK_STEP_MIX)):
        rc, ms, nbytes = hbm_probe_run(kind, [t.data_ptr() for t in bufs], quads, 3, reps, stream)
        if rc:
            raise RuntimeError(f"hbm_probe_run({name}) failed ({rc})")
        out[name] = round(nbytes / (ms * 1e-3) / 1e9, 1)
    for name, kind in (("first_mix_gbs", HBM_PROBE_FIRST_MIX), ("acc_mix_gbs", HBM_PROBE_ACC_MIX),
                       ("acc_mix_bulk_gbs", HBM_PROBE_BULK_ACC_MIX)):
        rc, ms, nbytes = hbm_probe_run(kind, [bufs[1].data_ptr(), bufs[0].data_ptr()], quads, 3, reps, stream)
        if rc:
            raise RuntimeError(f"hbm_probe_run({name}) failed ({rc})")
        out[name] = round(nbytes / (ms * 1e-3) / 1e9, 1)
    del bufs
    torch.cuda.empty_cache()
    return out
