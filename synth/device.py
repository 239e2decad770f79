"""Puts a workload's seeded inputs into torch device buffers (harness only).

Values are generated on the host by libsynth.so in slices, staged through a
pinned buffer and copied into the device tensor; nothing here computes any
part of the optimizer step.
"""
import numpy as np
import torch

from . import fill_grad, fill_master

SLICE = 1 << 26  # elements per staging slice


class Stager:
    """Reusable pinned staging buffers for uploads."""

    def __init__(self, slice_elems=SLICE):
        self.n = slice_elems
        self.h16 = torch.empty(slice_elems, dtype=torch.int16, pin_memory=True)
        self.h32 = torch.empty(slice_elems, dtype=torch.float32, pin_memory=True)

    def _upload(self, dst, first, fill, host):
        n = dst.numel()
        for off in range(0, n, self.n):
            k = min(self.n, n - off)
            buf = host[:k]
            arr = buf.numpy()
            if arr.dtype == np.int16:
                arr = arr.view(np.uint16)
            fill(arr, first + off)
            dst[off:off + k].copy_(buf, non_blocking=True)
            torch.cuda.current_stream().synchronize()

    def grad(self, wl, step, micro, dst, first=0):
        """dst (int16 device tensor) <- gradient elements [first, first+numel) of (step, micro)."""
        self._upload(dst, first, lambda a, f: fill_grad(wl, step, micro, a, f), self.h16)

    def master(self, wl, dst, first=0):
        """dst (float32 device tensor) <- initial masters [first, first+numel)."""
        self._upload(dst, first, lambda a, f: fill_master(wl, a, f), self.h32)


def host_grad(wl, step, micro, n=None, first=0):
    out = np.empty(wl.n if n is None else n, np.uint16)
    return fill_grad(wl, step, micro, out, first)


def host_master(wl, n=None, first=0):
    out = np.empty(wl.n if n is None else n, np.float32)
    return fill_master(wl, out, first)
