"""Page-locked host buffers for the end-to-end benchmark leg and its tests.

Harness plumbing, not part of the optimizer: the e2e measurement streams every
micro-batch gradient from host memory, and on the GPU host (a virtual machine)
how those host buffers are backed decides the copy rate.
"""
import ctypes
import mmap

import numpy as np
import torch


def _thp_size():
    """Size of a transparent huge page (512 MiB on 64 KiB-page Arm kernels, 2 MiB on 4 KiB ones)."""
    try:
        with open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size") as f:
            return int(f.read().strip())
    except (OSError, ValueError):
        return 2 << 20


def _huge_fraction(start, nbytes):
    """Fraction of [start, start + nbytes) backed by transparent huge pages (from /proc/self/smaps)."""
    try:
        huge, lo, hi = 0, None, None
        with open("/proc/self/smaps") as f:
            for line in f:
                head = line.split()[0]
                if "-" in head and ":" not in head:
                    lo, hi = (int(x, 16) for x in head.split("-"))
                elif head == "AnonHugePages:" and lo is not None and lo <= start < hi:
                    huge = int(line.split()[1]) * 1024
        return huge / nbytes if nbytes else 1.0
    except (OSError, ValueError):
        return 0.0


class PinnedHostBuffer:
    """Page-locked host memory for gradients that stream to the GPU.

    The region is aligned to the transparent-huge-page size and rounded up to
    whole huge pages, advised as huge (MADV_HUGEPAGE), faulted in and registered
    with cudaHostRegister.  Large pages keep the address translations of the
    host-to-device copies few: on a host whose memory is fragmented by earlier
    large jobs, small-page pinned buffers slowed copies that overlap HBM-bound
    kernels by almost 2x, huge-page ones far less.  Whole huge pages leave no
    small-page tail, which the kernel's background collapse (khugepaged) would
    keep trying, and failing, to merge while it is pinned.  `tensor` is a CPU
    tensor over the first numel elements (is_pinned()).  Falls back to the
    driver's pinned allocator (torch pin_memory) when the kernel cannot back at
    least 90 % of the region with huge pages (small-page registered memory was
    measured slower still) or registration is refused.
    """

    MADV_HUGEPAGE = 14

    def __init__(self, numel, dtype=torch.int16):
        itemsize = torch.empty(0, dtype=dtype).element_size()
        nbytes = int(numel) * itemsize
        self._registered = None
        self.huge_fraction = 0.0
        try:
            align = _thp_size()
            span = max(align, (nbytes + align - 1) // align * align)          # whole huge pages
            self._map = mmap.mmap(-1, span + align, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
            addr = ctypes.addressof(ctypes.c_char.from_buffer(self._map))
            start = (addr + align - 1) & ~(align - 1)
            libc = ctypes.CDLL(None, use_errno=True)
            libc.madvise.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
            libc.madvise(ctypes.c_void_p(start), span, self.MADV_HUGEPAGE)     # advisory
            whole = np.frombuffer(self._map, dtype=np.uint8, count=span, offset=start - addr)
            whole[:] = 0                                                        # fault every page in now
            self.huge_fraction = _huge_fraction(start, span)
            if self.huge_fraction < 0.9:
                raise RuntimeError("not backed by huge pages")
            if int(torch.cuda.cudart().cudaHostRegister(start, span, 0)) != 0:
                raise RuntimeError("cudaHostRegister refused")
            self._registered = start
            self.tensor = torch.from_numpy(whole[:nbytes]).view(dtype)
            self.huge_pages = True
        except Exception:
            self._map = None
            self.tensor = torch.empty(int(numel), dtype=dtype, pin_memory=True)
            self.huge_pages = False

    def close(self):
        """Unregister the region (the tensor must not be used afterwards)."""
        if self._registered is not None:
            torch.cuda.synchronize()
            torch.cuda.cudart().cudaHostUnregister(self._registered)
            self._registered = None
        self.tensor = None


def _h2d_gbs(src, dst, reps=2):
    """Best host-to-device copy rate (GB/s) of pinned `src` into device `dst`
    over `reps` whole-buffer copies on a side stream (the first may pay for
    lazy mappings)."""
    s = torch.cuda.Stream(dst.device)
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            dst[:src.numel()].copy_(src, non_blocking=True)
            e1.record(s)
        e1.synchronize()
        best = max(best, src.numel() * src.element_size() / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    return best


def fast_pinned_buffers(numel, count, dst, dtype=torch.int16, min_gbs=150.0, max_extra=12):
    """`count` PinnedHostBuffers of `numel` elements chosen by their measured
    host-to-device copy rate into the device tensor `dst` (at least numel
    elements; its contents are overwritten).  On a virtual machine the DMA rate
    of pinned host memory depends on how the hypervisor backs each region:
    3.4 GB buffers pinned side by side in one process copied at 211 GB/s or at
    12-136 GB/s.  A buffer below `min_gbs` is kept aside (so its memory is not
    handed out again at once) and another is pinned, up to `max_extra` extra
    buffers; the fastest `count` are kept and the rest freed.
    Returns (buffers, their rates in GB/s, number rejected)."""
    got, tries = [], 0
    while True:
        hb = PinnedHostBuffer(numel, dtype)
        got.append((_h2d_gbs(hb.tensor, dst), hb))
        fast = sum(1 for r, _ in got if r >= min_gbs)
        if fast >= count or len(got) >= count + max_extra:
            break
        tries += 1
    got.sort(key=lambda x: -x[0])
    keep, drop = got[:count], got[count:]
    for _, hb in drop:
        hb.close()
    return [hb for _, hb in keep], [round(r, 1) for r, _ in keep], len(drop)
