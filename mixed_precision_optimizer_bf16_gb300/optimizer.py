"""BF16Optimizer: drives the bf16opt C ABI from torch device tensors.

Marshalling only (data_ptr()s, stream handles, status -> exception); all
arithmetic is in libbf16opt.so.  State layout for one rank's shard:

  FLAT: master, exp_avg, exp_avg_sq, grad_accum (FP32) and param_bf16 (bf16)
        as five contiguous buffers of n elements, plus group ranges;
  LIST: the same five buffers per tensor (separate allocations).
"""
import contextlib

import torch

from . import bf16opt as C


def _ptr(t):
    return t.data_ptr() if t is not None else 0


_BF16_BITS = tuple(d for d in (torch.bfloat16, torch.int16, getattr(torch, "uint16", None)) if d is not None)


def _check_buffer(t, what, dtypes, numel=None):
    """A device tensor the library may read/write through a raw pointer: CUDA,
    contiguous, one of `dtypes`, and `numel` elements when given.  The C ABI
    receives bare pointers and cannot check any of this itself."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{what}: must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{what}: dtype {t.dtype}, expected one of {[str(d) for d in dtypes]}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{what}: {t.numel()} elements, expected {numel}")


def _check_state(d, what, offload=False):
    n = d["master"].numel()
    for k in ("master", "exp_avg", "exp_avg_sq", "grad_accum"):
        if offload and k != "grad_accum":
            _check_host_buffer(d[k], f"{what}[{k!r}]", n)
        else:
            _check_buffer(d[k], f"{what}[{k!r}]", (torch.float32,), n)
    _check_buffer(d["param_bf16"], f"{what}['param_bf16']", _BF16_BITS, n)
    return n


def _check_host_buffer(t, what, numel):
    """An FP32 host tensor the library's host threads read and write (offload)."""
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError(f"{what}: must be a CPU tensor (offloaded state)")
    if t.dtype != torch.float32 or not t.is_contiguous() or t.numel() != numel:
        raise ValueError(f"{what}: must be a contiguous float32 tensor of {numel} elements")


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def alloc_flat(n, device="cuda", misalign=0):
    """Five state buffers of n elements; each starts `misalign` elements past
    a 256-byte boundary (the allocator's own alignment is at least that)."""
    def one(dtype):
        base = torch.empty(n + misalign + 64, dtype=dtype, device=device)
        assert base.data_ptr() % 256 == 0
        return base[misalign:misalign + n]
    return dict(master=one(torch.float32), exp_avg=one(torch.float32), exp_avg_sq=one(torch.float32),
                grad_accum=one(torch.float32), param_bf16=one(torch.int16))


def resident_pattern(gas, fold=8):
    """Per-micro-batch `defer` flags for a step whose micro-batch gradients all
    stay resident (one buffer each): all deferred when gas <= fold (the FP32
    accumulator is never stored); otherwise runs of `fold`, each folded into
    the accumulator by its last micro-batch, and the final run deferred into
    the norm pass and the step -- never more than `fold` pending, the library's
    limit (8).  At GAS 32: 134 instead of 344 bytes per element per step."""
    if gas <= fold:
        return [True] * gas
    tail = gas % fold or fold
    head = gas - tail
    return [(k % fold) != fold - 1 for k in range(head)] + [True] * tail


def gather_sumsqs(local, group=None):
    """Every rank's local sum of squares, in rank order (an all-gather of one
    FP64 scalar per rank); [local] when torch.distributed is not initialised.
    Only moves the values: the library sums them (bf16opt_set_rank_sumsqs)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return [float(local)]
    world = dist.get_world_size(group)
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    mine = torch.tensor([float(local)], dtype=torch.float64, device=dev)
    parts = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine, group=group)
    return [float(p.item()) for p in parts]


def partition_bounds(n, world):
    """ZeRO flat partitioning: rank r owns elements [b[r], b[r+1]) of the n
    elements of the flat buffer, contiguous slices of ceil(n / world) elements
    (the last ones shorter or empty)."""
    part = -(-int(n) // int(world)) if world > 0 else 0
    return [min(int(n), r * part) for r in range(int(world) + 1)]


def exchange_gradient_slices(full_grad, bounds, group=None, phase=0):
    """The exchange half of a ZeRO-2 gradient reduce-scatter.

    full_grad: this rank's bf16 gradient (bf16 or int16 tensor) of the whole
    flat buffer; bounds: partition_bounds(n, world).  Every rank sends
    partition p of its gradient to rank p and receives its own partition from
    every rank.  Returns a tensor [world, own partition size] on full_grad's
    device: row q is rank q's gradient over this rank's partition, so the rows
    are in rank order.  Point-to-point sends of byte views (gloo has no
    all-to-all and no 16-bit types); with gloo a CUDA gradient is staged
    through host memory.  phase: element offset (0-31) of every row within a
    128-byte line -- give the accumulator's, so that the library streams rows
    and accumulator as aligned vectors.  Without an initialised process group
    the only row is the gradient itself."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return full_grad.reshape(1, -1)
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    if len(bounds) != world + 1 or bounds[-1] != full_grad.numel():
        raise ValueError("bounds must be partition_bounds(full_grad.numel(), world)")
    stage = full_grad.is_cuda and dist.get_backend(group) != "nccl"
    src = full_grad.detach().cpu() if stage else full_grad.detach()
    src = src.contiguous().view(torch.uint8)
    lo, hi = bounds[rank], bounds[rank + 1]
    # rows of whole 128-byte lines (the allocation starts on one), each row's
    # elements starting `phase` elements into its first line
    ph = int(phase) % 32
    stride = -(-(hi - lo + ph) // 64) * 64
    out = torch.empty((world, max(stride, 1)), dtype=full_grad.dtype, device=full_grad.device)
    recv = torch.empty_like(out, device="cpu") if stage else out
    ops = []
    for q in range(world):
        peer = dist.get_global_rank(group, q) if group is not None else q
        if q == rank:
            recv[q, ph:ph + hi - lo].view(torch.uint8).copy_(src[2 * lo:2 * hi])
            continue
        if bounds[q + 1] > bounds[q]:
            ops.append(dist.P2POp(dist.isend, src[2 * bounds[q]:2 * bounds[q + 1]], peer, group))
        if hi > lo:
            ops.append(dist.P2POp(dist.irecv, recv[q, ph:ph + hi - lo].view(torch.uint8), peer, group))
    if ops:
        for w in dist.batch_isend_irecv(ops):
            w.wait()
    if stage:
        out.copy_(recv)
    return out[:, ph:ph + hi - lo]


def fold_pattern(slices, last):
    """Deferral flags for folding `slices` received gradient slices of one
    micro-batch: every run of 8 is folded by its 8th (the library keeps at most
    8 pending); within the last micro-batch the final run stays deferred into
    the norm pass and the step, otherwise the final slice folds it."""
    flags = resident_pattern(slices)
    if not last:
        flags[-1] = False
    return flags


class BF16Optimizer:
    """One handle over a FLAT shard (`flat` = dict of the five tensors, `ranges`)
    or a LIST of tensors (`tensors` = list of such dicts with a "group" key)."""

    def __init__(self, groups, flat=None, ranges=None, tensors=None, max_grad_norm=1.0, grad_scale=1.0,
                 offload=False, offload_threads=0):
        """offload=True (FLAT only): ZeRO-Offload -- flat master, exp_avg and
        exp_avg_sq are CPU tensors updated by offload_threads host threads
        (0: one per core); grad_accum and param_bf16 stay on the GPU."""
        if (flat is None) == (tensors is None):
            raise ValueError("give exactly one of flat= or tensors=")
        if offload and flat is None:
            raise ValueError("offload needs a FLAT shard (flat=)")
        self.groups = [dict(g) for g in groups]
        self.offload = bool(offload)
        if flat is not None:
            n = _check_state(flat, "flat", offload=self.offload)
            self.n, self.numels = n, None
            self.desc = C.flat_desc(n, _ptr(flat["master"]), _ptr(flat["exp_avg"]), _ptr(flat["exp_avg_sq"]),
                                    _ptr(flat["grad_accum"]), _ptr(flat["param_bf16"]), self.groups, ranges,
                                    max_grad_norm, grad_scale)
            self.mode = C.BF16OPT_FLAT
        else:
            self.n, self.numels = None, [_check_state(t, f"tensors[{i}]") for i, t in enumerate(tensors)]
            tl = [(_ptr(t["master"]), _ptr(t["exp_avg"]), _ptr(t["exp_avg_sq"]), _ptr(t["grad_accum"]),
                   _ptr(t["param_bf16"]), t["master"].numel(), int(t.get("group", 0))) for t in tensors]
            self.desc = C.list_desc(tl, self.groups, max_grad_norm, grad_scale)
            self.mode = C.BF16OPT_LIST
        # the library holds raw pointers: keep the tensors alive with the handle
        self._state = [flat] if flat is not None else list(tensors)
        self._sched_args = None
        self._skip = False
        if self.offload:
            rc, self.h = C.bf16opt_create_offload(self.desc, offload_threads)
        else:
            rc, self.h = C.bf16opt_create(self.desc)
        C.check(rc, None)

    @classmethod
    def from_parameters(cls, param_groups, lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.0,
                        max_grad_norm=1.0, grad_scale=1.0, grad_buffers=1):
        """One FLAT shard over a model's bf16 parameters.

        param_groups: an iterable of parameters, or torch.optim-style dicts
        {"params": [...], optional "lr", "betas", "eps", "weight_decay"}.  Every
        parameter must be a bf16 CUDA tensor.  The parameters are laid out one
        after another, group by group (one range per group); the FP32 masters
        start as the parameters' values; afterwards each parameter's .data is a
        view into the flat bf16 parameter buffer (the step writes it in place)
        and its .grad a view into the flat bf16 gradient buffer `grad_buffer`,
        which backward adds into: call zero_grad() before each micro-batch's
        backward and accumulate() (no gradient argument) after it.

        grad_buffers=N allocates N flat gradient buffers (2 bytes per element
        each); use_grad_buffer(i) points every .grad at buffer i.  With one
        buffer per micro-batch every micro-batch can be deferred, so the FP32
        accumulator is never stored: 42 instead of 64 bytes per element per
        step at GAS 4, the same FP32 adds in the same order.
        """
        groups = list(param_groups)
        if groups and isinstance(groups[0], torch.Tensor):
            groups = [{"params": groups}]
        seen, layout, hyper, ranges, n = set(), [], [], [], 0
        for gi, g in enumerate(groups):
            b1, b2 = g.get("betas", betas)
            hyper.append(dict(lr=float(g.get("lr", lr)), beta1=float(b1), beta2=float(b2), eps=float(g.get("eps", eps)),
                              weight_decay=float(g.get("weight_decay", weight_decay))))
            begin = n
            for p in g["params"]:
                if id(p) in seen:
                    raise ValueError("a parameter appears twice")
                if not (isinstance(p, torch.Tensor) and p.is_cuda and p.dtype == torch.bfloat16):
                    raise ValueError("every parameter must be a bf16 CUDA tensor")
                seen.add(id(p))
                layout.append((p, n))
                n += p.numel()
            ranges.append((begin, n, gi))
        dev = layout[0][0].device if layout else torch.device("cuda")
        flat = {k: torch.zeros(n, dtype=torch.float32, device=dev)
                for k in ("master", "exp_avg", "exp_avg_sq", "grad_accum")}
        flat["param_bf16"] = torch.empty(n, dtype=torch.bfloat16, device=dev)
        if grad_buffers < 1:
            raise ValueError("grad_buffers must be >= 1")
        bufs = [torch.zeros(n, dtype=torch.bfloat16, device=dev) for _ in range(int(grad_buffers))]
        with torch.no_grad():
            for p, off in layout:
                k = p.numel()
                flat["param_bf16"][off:off + k].copy_(p.reshape(-1))
                flat["master"][off:off + k].copy_(p.reshape(-1).float())
                p.data = flat["param_bf16"][off:off + k].view(p.shape)
        opt = cls(hyper, flat=flat, ranges=ranges, max_grad_norm=max_grad_norm, grad_scale=grad_scale)
        opt.flat = flat
        opt.ranges = ranges
        opt.grad_buffers = bufs
        opt._layout = layout
        opt.use_grad_buffer(0)
        return opt

    def use_grad_buffer(self, i, stream=None):
        """Point every parameter's .grad at flat gradient buffer i of a
        from_parameters() optimizer and zero that buffer; returns it."""
        buf = self.grad_buffers[i]
        for p, off in self._layout:
            p.grad = buf[off:off + p.numel()].view(p.shape)
        self.grad_buffer = buf
        self.zero_grad(stream)
        return buf

    def zero_grad(self, stream=None):
        """Zero the current flat gradient buffer of a from_parameters() optimizer."""
        with torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext():
            self.grad_buffer.zero_()

    def accumulate(self, grad=None, first=False, last=False, defer=False, stream=None):
        """grad: bf16 (or int16-viewed) tensor (FLAT) or list of them (LIST);
        None = the flat gradient buffer of a from_parameters() optimizer."""
        if grad is None:
            grad = getattr(self, "grad_buffer", None)
            if grad is None:
                raise ValueError("no gradient given and no gradient buffer (see from_parameters)")
        flags = (C.BF16OPT_FIRST if first else 0) | (C.BF16OPT_LAST if last else 0) | (C.BF16OPT_DEFER if defer else 0)
        if self.mode == C.BF16OPT_FLAT:
            if self.n:
                _check_buffer(grad, "grad", _BF16_BITS, self.n)
            rc = C.bf16opt_accumulate(self.h, _ptr(grad) if self.n else 0, None, flags, _stream_handle(stream))
        else:
            if len(grad) != len(self.numels):
                raise ValueError(f"grad: {len(grad)} tensors, expected {len(self.numels)}")
            for i, (g, k) in enumerate(zip(grad, self.numels)):
                if k:
                    _check_buffer(g, f"grad[{i}]", _BF16_BITS, k)
            rc = C.bf16opt_accumulate(self.h, 0, [_ptr(g) if k else 0 for g, k in zip(grad, self.numels)], flags,
                                      _stream_handle(stream))
        return C.check(rc, self.h)

    def accumulate_reduce_scatter(self, full_grad, first=False, last=False, group=None, stream=None):
        """ZeRO-2 gradient reduction feeding the FP32 accumulation.

        This optimizer holds one rank's partition (FLAT) of a flat buffer split
        by partition_bounds; full_grad is this rank's bf16 gradient of the whole
        buffer for one micro-batch.  The partitions are exchanged
        (exchange_gradient_slices) and the world received slices of this
        rank's partition are folded into the FP32 accumulator in rank order --
        one FP32 add per slice, micro-batch by micro-batch, rank by rank, the
        same arithmetic as accumulating them as consecutive micro-batches.
        The slices ride on DEFER (runs of at most 8 folded in one pass); those
        of the last micro-batch stay deferred until the step, which keeps the
        received buffer alive until then.  first/last: as for accumulate()."""
        import torch.distributed as dist
        if self.mode != C.BF16OPT_FLAT:
            raise ValueError("accumulate_reduce_scatter needs a FLAT partition")
        world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
        bounds = partition_bounds(full_grad.numel(), world)
        rank = dist.get_rank(group) if world > 1 else 0
        if bounds[rank + 1] - bounds[rank] != self.n:
            raise ValueError(f"partition of rank {rank} has {bounds[rank + 1] - bounds[rank]} elements, "
                             f"this optimizer {self.n}")
        # rows at the accumulator's element offset within a 128-byte line
        phase = (self._state[0]["grad_accum"].data_ptr() // 4) % 32 if self.n else 0
        with torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext():
            recv = exchange_gradient_slices(full_grad, bounds, group, phase)
        flags = fold_pattern(world, last)
        for q in range(world):
            self.accumulate(recv[q], first=first and q == 0, last=last and q == world - 1, defer=flags[q],
                            stream=stream)
        # deferred slices are read by a later pass: keep their buffer until then
        self._recv_alive = recv if any(flags) else None
        return recv

    def grad_norm(self, stream=None, sync=False):
        rc, norm = C.bf16opt_grad_norm(self.h, _stream_handle(stream), want_norm=sync)
        C.check(rc, self.h)
        return norm

    def grad_norm_distributed(self, group=None, stream=None):
        """Global norm over every rank's partition: this rank's FP64 sum of squares
        is all-gathered; the library sums the gathered values in rank order
        (the same bits on every rank) and sets the norm and clip coefficient.
        Returns the global norm the library computed."""
        import torch.distributed as dist
        rc, local = C.bf16opt_grad_norm_local(self.h, _stream_handle(stream))
        C.check(rc, self.h)
        parts = gather_sumsqs(local, group)
        rank = dist.get_rank(group) if dist.is_available() and dist.is_initialized() else 0
        rc, norm = C.bf16opt_set_rank_sumsqs(self.h, parts, rank, _stream_handle(stream))
        C.check(rc, self.h)
        return norm

    def set_skip_nonfinite(self, enable=True):
        """Skip (on the device) any step whose global norm is Inf or NaN."""
        rc = C.check(C.bf16opt_set_skip_nonfinite(self.h, enable), self.h)
        self._skip = bool(enable)
        return rc

    def set_lr_schedule(self, warmup_steps, decay_steps, min_lr_ratio):
        """Attach the warmup + cosine schedule (None detaches); see bf16opt_set_lr_schedule."""
        self._sched = None if warmup_steps is None else C.lr_schedule(warmup_steps, decay_steps, min_lr_ratio)
        rc = C.check(C.bf16opt_set_lr_schedule(self.h, self._sched), self.h)
        self._sched_args = None if warmup_steps is None else (int(warmup_steps), int(decay_steps), float(min_lr_ratio))
        return rc

    _CKPT_KEYS = ("master", "exp_avg", "exp_avg_sq", "param_bf16")

    def state_dict(self):
        """Checkpoint: the step counter, the settings and host copies of every
        tensor's FP32 master, moments and bf16 parameters (the accumulator carries
        nothing between steps).  Waits for the device (the step counter read does)."""
        t = self.t
        return {"t": t, "groups": [dict(g) for g in self.groups], "lr_schedule": self._sched_args,
                "skip_nonfinite": self._skip,
                "tensors": [{k: d[k].detach().to("cpu", copy=True) for k in self._CKPT_KEYS} for d in self._state]}

    def load_state_dict(self, sd):
        """Restore a state_dict() into this optimizer's buffers (same layout:
        tensor count, sizes and dtypes) and continue from its step.  Continuing
        is bit-identical to an uninterrupted run when every buffer has the same
        offset modulo 128 bytes as when the checkpoint was taken (that offset
        fixes the chunking of the norm's partial sums)."""
        if len(sd["tensors"]) != len(self._state):
            raise ValueError(f"checkpoint has {len(sd['tensors'])} tensors, this optimizer {len(self._state)}")
        if [dict(g) for g in sd["groups"]] != self.groups:
            raise ValueError("checkpoint groups differ from this optimizer's")
        for i, (src, dst) in enumerate(zip(sd["tensors"], self._state)):
            for k in self._CKPT_KEYS:
                if src[k].shape != dst[k].shape or src[k].element_size() != dst[k].element_size():
                    raise ValueError(f"tensors[{i}][{k!r}]: checkpoint {tuple(src[k].shape)}/{src[k].dtype}, "
                                     f"buffer {tuple(dst[k].shape)}/{dst[k].dtype}")
        torch.cuda.synchronize()
        for src, dst in zip(sd["tensors"], self._state):
            for k in self._CKPT_KEYS:
                dst[k].copy_(src[k].view(dst[k].dtype))
        torch.cuda.synchronize()
        if sd.get("lr_schedule") is not None:
            self.set_lr_schedule(*sd["lr_schedule"])
        self.set_skip_nonfinite(bool(sd.get("skip_nonfinite", False)))
        self.t = int(sd["t"])

    def step(self, lr=None, stream=None):
        """lr: None (the groups' rates), one rate for every group, or one per group."""
        lrs = None if lr is None else ([float(lr)] * len(self.groups) if not hasattr(lr, "__len__") else list(lr))
        if lrs is not None and len(lrs) != len(self.groups):
            raise ValueError(f"lr: {len(lrs)} rates for {len(self.groups)} groups")
        rc = C.check(C.bf16opt_step(self.h, lrs, _stream_handle(stream)), self.h)
        # received gradient slices the step folded may be freed once it has run
        # (the caching allocator reuses them in stream order)
        self._recv_alive = None
        return rc

    @property
    def t(self):
        rc, t = C.bf16opt_get_step(self.h)
        C.check(rc, self.h)
        return t

    @t.setter
    def t(self, value):
        C.check(C.bf16opt_set_step(self.h, value), self.h)

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            C.bf16opt_destroy(self.h)
            self.h = None
        self._state = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
