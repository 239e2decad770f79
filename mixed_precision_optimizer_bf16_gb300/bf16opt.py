"""Python binding of libbf16opt.so: the C ABI of include/bf16opt.h, same names.

Argument marshalling only.  Every step of the optimizer runs in the library's
CUDA kernels; there is no Python or CPU fallback, and loading fails loudly
when the library has not been built.  Device memory and streams may come
from PyTorch: pass `tensor.data_ptr()` and `stream.cuda_stream` (ints).
"""
import ctypes
import os

from . import build as _build

BF16OPT_OK = 0
BF16OPT_WARN_NONFINITE = 1
BF16OPT_ERR_INVALID_ARG = -1
BF16OPT_ERR_ALIGNMENT = -2
BF16OPT_ERR_SEQUENCE = -3
BF16OPT_ERR_OOM = -4
BF16OPT_ERR_CUDA = -5
BF16OPT_ERR_UNSUPPORTED = -6

BF16OPT_FLAT = 0
BF16OPT_LIST = 1
BF16OPT_FIRST = 1
BF16OPT_LAST = 2
BF16OPT_DEFER = 4
BF16OPT_MAX_GROUPS = 16
BF16OPT_MAX_DEFERRED = 8
BF16OPT_STATIC_NORM_MAX_ELEMS = 1 << 30
BF16OPT_PATH_NONE = 0
BF16OPT_PATH_VECTOR = 1
BF16OPT_PATH_PIPELINE = 2
BF16OPT_PATH_HOST = 3

c_u64, c_u32, c_i32, c_f32, c_vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p


class bf16opt_range_t(ctypes.Structure):
    _fields_ = [("begin", c_u64), ("end", c_u64), ("group", c_u32), ("reserved", c_u32)]


class bf16opt_tensor_t(ctypes.Structure):
    _fields_ = [("master", c_vp), ("exp_avg", c_vp), ("exp_avg_sq", c_vp), ("grad_accum", c_vp),
                ("param_bf16", c_vp), ("numel", c_u64), ("group", c_u32), ("reserved", c_u32)]


class bf16opt_group_t(ctypes.Structure):
    _fields_ = [("lr", c_f32), ("beta1", c_f32), ("beta2", c_f32), ("eps", c_f32), ("weight_decay", c_f32)]


class bf16opt_desc_t(ctypes.Structure):
    _fields_ = [("mode", c_i32), ("n_groups", c_u32), ("groups", ctypes.POINTER(bf16opt_group_t)),
                ("n", c_u64), ("master", c_vp), ("exp_avg", c_vp), ("exp_avg_sq", c_vp), ("grad_accum", c_vp),
                ("param_bf16", c_vp), ("ranges", ctypes.POINTER(bf16opt_range_t)), ("n_ranges", c_u32),
                ("n_tensors", c_u32), ("tensors", ctypes.POINTER(bf16opt_tensor_t)),
                ("max_grad_norm", c_f32), ("grad_scale", c_f32)]


class bf16opt_lr_schedule_t(ctypes.Structure):
    _fields_ = [("warmup_steps", ctypes.c_int64), ("decay_steps", ctypes.c_int64), ("min_lr_ratio", c_f32),
                ("reserved", c_u32)]


class bf16opt_norm_result_t(ctypes.Structure):
    _fields_ = [("sumsq", ctypes.c_double), ("norm", ctypes.c_double), ("clip_coef", ctypes.c_double)]


# Functions the header declares (the tests check the library exports them all).
EXPORTS = ("bf16opt_create", "bf16opt_create_offload", "bf16opt_accumulate", "bf16opt_grad_norm", "bf16opt_step", "bf16opt_destroy",
           "bf16opt_get_step", "bf16opt_set_step", "bf16opt_error_string", "bf16opt_last_error",
           "bf16opt_grad_norm_static", "bf16opt_lr_factor", "bf16opt_set_lr_schedule",
           "bf16opt_grad_norm_local", "bf16opt_set_global_sumsq", "bf16opt_set_rank_sumsqs",
           "bf16opt_sum_rank_sumsqs", "bf16opt_set_skip_nonfinite", "bf16opt_debug_faults",
           "bf16opt_pipeline_timeouts", "bf16opt_step_path", "bf16opt_abi_version")

ABI_VERSION = 2   # BF16OPT_ABI_VERSION of the header these declarations mirror

_lib = None


def lib_path():
    """The library to load: $BF16OPT_LIBRARY if set (e.g. a checked build of the
    same sources), else the in-tree libbf16opt.so."""
    return os.environ.get("BF16OPT_LIBRARY") or _build.LIB_PATH


def load(path=None):
    """Load libbf16opt.so (built by __graft_entry__.build() or build.build())."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libbf16opt.so is not built ({path}); run __graft_entry__.build() -- "
                           "there is no fallback implementation")
    L = ctypes.CDLL(path)
    L.bf16opt_abi_version.restype = ctypes.c_int
    L.bf16opt_abi_version.argtypes = []
    if L.bf16opt_abi_version() != ABI_VERSION:
        raise RuntimeError(f"{path} has ABI version {L.bf16opt_abi_version()}, this binding {ABI_VERSION}: rebuild")
    hp = ctypes.c_void_p
    L.bf16opt_create.restype = ctypes.c_int
    L.bf16opt_create.argtypes = [ctypes.POINTER(bf16opt_desc_t), ctypes.POINTER(hp)]
    L.bf16opt_create_offload.restype = ctypes.c_int
    L.bf16opt_create_offload.argtypes = [ctypes.POINTER(bf16opt_desc_t), ctypes.c_int, ctypes.POINTER(hp)]
    L.bf16opt_accumulate.restype = ctypes.c_int
    L.bf16opt_accumulate.argtypes = [hp, c_vp, ctypes.POINTER(c_vp), ctypes.c_uint, c_vp]
    L.bf16opt_grad_norm.restype = ctypes.c_int
    L.bf16opt_grad_norm.argtypes = [hp, c_vp, ctypes.POINTER(ctypes.c_double)]
    L.bf16opt_step.restype = ctypes.c_int
    L.bf16opt_step.argtypes = [hp, ctypes.POINTER(c_f32), c_vp]
    L.bf16opt_destroy.restype = ctypes.c_int
    L.bf16opt_destroy.argtypes = [hp]
    L.bf16opt_get_step.restype = ctypes.c_int
    L.bf16opt_get_step.argtypes = [hp, ctypes.POINTER(ctypes.c_int64)]
    L.bf16opt_set_step.restype = ctypes.c_int
    L.bf16opt_set_step.argtypes = [hp, ctypes.c_int64]
    L.bf16opt_error_string.restype = ctypes.c_char_p
    L.bf16opt_error_string.argtypes = [ctypes.c_int]
    L.bf16opt_last_error.restype = ctypes.c_char_p
    L.bf16opt_last_error.argtypes = [hp]
    L.bf16opt_grad_norm_local.restype = ctypes.c_int
    L.bf16opt_grad_norm_local.argtypes = [hp, c_vp, ctypes.POINTER(ctypes.c_double)]
    L.bf16opt_set_global_sumsq.restype = ctypes.c_int
    L.bf16opt_set_global_sumsq.argtypes = [hp, ctypes.c_double, c_vp]
    L.bf16opt_set_rank_sumsqs.restype = ctypes.c_int
    L.bf16opt_set_rank_sumsqs.argtypes = [hp, ctypes.POINTER(ctypes.c_double), c_u32, c_u32, c_vp,
                                          ctypes.POINTER(ctypes.c_double)]
    L.bf16opt_sum_rank_sumsqs.restype = ctypes.c_int
    L.bf16opt_sum_rank_sumsqs.argtypes = [ctypes.POINTER(ctypes.c_double), c_u32, ctypes.POINTER(ctypes.c_double)]
    L.bf16opt_set_skip_nonfinite.restype = ctypes.c_int
    L.bf16opt_set_skip_nonfinite.argtypes = [hp, ctypes.c_int]
    L.bf16opt_debug_faults.restype = ctypes.c_int
    L.bf16opt_debug_faults.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.bf16opt_pipeline_timeouts.restype = ctypes.c_int
    L.bf16opt_step_path.restype = ctypes.c_int
    L.bf16opt_step_path.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    L.bf16opt_pipeline_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.bf16opt_lr_factor.restype = ctypes.c_int
    L.bf16opt_lr_factor.argtypes = [ctypes.POINTER(bf16opt_lr_schedule_t), ctypes.c_int64,
                                    ctypes.POINTER(ctypes.c_double)]
    L.bf16opt_set_lr_schedule.restype = ctypes.c_int
    L.bf16opt_set_lr_schedule.argtypes = [hp, ctypes.POINTER(bf16opt_lr_schedule_t)]
    L.bf16opt_grad_norm_static.restype = ctypes.c_int
    L.bf16opt_grad_norm_static.argtypes = [c_vp, c_u64, c_f32, c_f32, c_vp, c_vp]
    if path == lib_path():
        _lib = L
    return L


# ---- same-name wrappers (return the C status; outputs as extra return values)

def bf16opt_create(desc):
    h = ctypes.c_void_p()
    rc = load().bf16opt_create(ctypes.byref(desc), ctypes.byref(h))
    return rc, h


def bf16opt_create_offload(desc, n_threads=0):
    """FLAT descriptor whose master and moments are host addresses (ZeRO-Offload)."""
    h = ctypes.c_void_p()
    rc = load().bf16opt_create_offload(ctypes.byref(desc), int(n_threads), ctypes.byref(h))
    return rc, h


def bf16opt_accumulate(h, grad_flat, grad_list, flags, stream=0):
    arr = None
    if grad_list is not None:
        arr = (c_vp * len(grad_list))(*[c_vp(int(p)) for p in grad_list])
    return load().bf16opt_accumulate(h, c_vp(int(grad_flat)) if grad_flat else None, arr, flags,
                                     c_vp(int(stream)) if stream else None)


def bf16opt_grad_norm(h, stream=0, want_norm=False):
    out = ctypes.c_double(0.0)
    rc = load().bf16opt_grad_norm(h, c_vp(int(stream)) if stream else None,
                                  ctypes.byref(out) if want_norm else None)
    return rc, (out.value if want_norm else None)


def bf16opt_step(h, lr_override=None, stream=0):
    arr = None
    if lr_override is not None:
        arr = (c_f32 * len(lr_override))(*lr_override)
    return load().bf16opt_step(h, arr, c_vp(int(stream)) if stream else None)


def bf16opt_destroy(h):
    return load().bf16opt_destroy(h)


def bf16opt_get_step(h):
    t = ctypes.c_int64(0)
    rc = load().bf16opt_get_step(h, ctypes.byref(t))
    return rc, t.value


def bf16opt_set_step(h, t):
    return load().bf16opt_set_step(h, int(t))


def bf16opt_grad_norm_local(h, stream=0):
    out = ctypes.c_double(0.0)
    rc = load().bf16opt_grad_norm_local(h, c_vp(int(stream)) if stream else None, ctypes.byref(out))
    return rc, out.value


def bf16opt_set_global_sumsq(h, global_sumsq, stream=0):
    return load().bf16opt_set_global_sumsq(h, float(global_sumsq), c_vp(int(stream)) if stream else None)


def bf16opt_set_rank_sumsqs(h, per_rank, rank, stream=0):
    """per_rank: every rank's local sum of squares, in rank order.  Returns (status, global norm)."""
    arr = (ctypes.c_double * max(1, len(per_rank)))(*[float(x) for x in per_rank])
    norm = ctypes.c_double(0.0)
    rc = load().bf16opt_set_rank_sumsqs(h, arr if len(per_rank) else None, len(per_rank), int(rank),
                                        c_vp(int(stream)) if stream else None, ctypes.byref(norm))
    return rc, norm.value


def bf16opt_sum_rank_sumsqs(per_rank):
    """Returns (status, the rank-ordered FP64 sum)."""
    arr = (ctypes.c_double * max(1, len(per_rank)))(*[float(x) for x in per_rank])
    out = ctypes.c_double(0.0)
    rc = load().bf16opt_sum_rank_sumsqs(arr if len(per_rank) else None, len(per_rank), ctypes.byref(out))
    return rc, out.value


def bf16opt_set_skip_nonfinite(h, enable):
    return load().bf16opt_set_skip_nonfinite(h, 1 if enable else 0)


def bf16opt_lr_factor(sched, t):
    f = ctypes.c_double(0.0)
    rc = load().bf16opt_lr_factor(ctypes.byref(sched) if sched is not None else None, int(t), ctypes.byref(f))
    return rc, f.value


def bf16opt_set_lr_schedule(h, sched):
    return load().bf16opt_set_lr_schedule(h, ctypes.byref(sched) if sched is not None else None)


def lr_schedule(warmup_steps, decay_steps, min_lr_ratio):
    return bf16opt_lr_schedule_t(int(warmup_steps), int(decay_steps), float(min_lr_ratio), 0)


def bf16opt_grad_norm_static(grad_accum, n, grad_scale, max_grad_norm, out, stream=0):
    """grad_accum, out: device addresses (ints); out receives a bf16opt_norm_result_t.
    Allocates nothing (its scratch is a fixed static device array)."""
    return load().bf16opt_grad_norm_static(c_vp(int(grad_accum)) if grad_accum else None, n, grad_scale,
                                           max_grad_norm, c_vp(int(out)) if out else None,
                                           c_vp(int(stream)) if stream else None)


def bf16opt_error_string(code):
    return load().bf16opt_error_string(code).decode()


def bf16opt_debug_faults():
    """(status, fault bits) of a checked build; release builds give UNSUPPORTED."""
    bits = ctypes.c_uint32(0)
    rc = load().bf16opt_debug_faults(ctypes.byref(bits))
    return rc, bits.value


def bf16opt_pipeline_timeouts():
    """(status, waits of the step's copy pipeline that gave up since the last call)."""
    n = ctypes.c_uint32(0)
    rc = load().bf16opt_pipeline_timeouts(ctypes.byref(n))
    return rc, n.value


def bf16opt_step_path(h):
    """(status, BF16OPT_PATH_* of the handle's last step)."""
    path = ctypes.c_int(0)
    rc = load().bf16opt_step_path(h, ctypes.byref(path))
    return rc, path.value


def bf16opt_last_error(h=None):
    return load().bf16opt_last_error(h).decode()


# ---- descriptor helpers

def make_groups(groups):
    """groups: list of dicts with lr, beta1, beta2, eps, weight_decay."""
    arr = (bf16opt_group_t * len(groups))()
    for i, g in enumerate(groups):
        arr[i] = bf16opt_group_t(g["lr"], g["beta1"], g["beta2"], g["eps"], g["weight_decay"])
    return arr


def flat_desc(n, master, exp_avg, exp_avg_sq, grad_accum, param_bf16, groups, ranges=None,
              max_grad_norm=1.0, grad_scale=1.0):
    """FLAT descriptor from device addresses (ints).  Keep the returned object
    alive until bf16opt_create has returned (it owns the host arrays)."""
    g = make_groups(groups)
    d = bf16opt_desc_t()
    d.mode = BF16OPT_FLAT
    d.n_groups = len(groups)
    d.groups = ctypes.cast(g, ctypes.POINTER(bf16opt_group_t))
    d.n = n
    d.master, d.exp_avg, d.exp_avg_sq, d.grad_accum, d.param_bf16 = (
        c_vp(int(x)) if x else None for x in (master, exp_avg, exp_avg_sq, grad_accum, param_bf16))
    r = None
    if ranges:
        r = (bf16opt_range_t * len(ranges))(*[bf16opt_range_t(b, e, gi, 0) for b, e, gi in ranges])
        d.ranges = ctypes.cast(r, ctypes.POINTER(bf16opt_range_t))
        d.n_ranges = len(ranges)
    d.max_grad_norm = max_grad_norm
    d.grad_scale = grad_scale
    d._keep = (g, r)
    return d


def list_desc(tensors, groups, max_grad_norm=1.0, grad_scale=1.0):
    """LIST descriptor; tensors: list of (master, exp_avg, exp_avg_sq, grad_accum, param_bf16, numel, group)."""
    g = make_groups(groups)
    t = (bf16opt_tensor_t * max(1, len(tensors)))()
    for i, (p, m, v, a, b, n, gi) in enumerate(tensors):
        t[i] = bf16opt_tensor_t(c_vp(int(p)) if p else None, c_vp(int(m)) if m else None,
                                c_vp(int(v)) if v else None, c_vp(int(a)) if a else None,
                                c_vp(int(b)) if b else None, n, gi, 0)
    d = bf16opt_desc_t()
    d.mode = BF16OPT_LIST
    d.n_groups = len(groups)
    d.groups = ctypes.cast(g, ctypes.POINTER(bf16opt_group_t))
    d.n_tensors = len(tensors)
    d.tensors = ctypes.cast(t, ctypes.POINTER(bf16opt_tensor_t))
    d.max_grad_norm = max_grad_norm
    d.grad_scale = grad_scale
    d._keep = (g, t)
    return d


class Bf16OptError(RuntimeError):
    def __init__(self, rc, msg):
        super().__init__(f"{bf16opt_error_string(rc)} ({rc}): {msg}")
        self.rc = rc


def check(rc, h=None):
    if rc < 0:
        raise Bf16OptError(rc, bf16opt_last_error(h))
    return rc
