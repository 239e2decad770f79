"""Parity harness: the CUDA path (through the C ABI) against the CPU oracle.

GPU side: a workload's shard lives in torch device buffers; seeded inputs are
written by the device generator (synth.gpu, bit-identical to the host one);
every optimizer call goes through libbf16opt.so.
Oracle side: the same inputs regenerated on the host; either a dense run over
the whole shard, or (for shards too large to materialise) the global norm of
every step streamed from the counters plus whole-run replays of sampled
elements.

Tolerances (the workload definitions' bar, plainest reading where silent):
  accumulator    bit-exact;
  global norm    |n_gpu - n_ref| <= 1e-6 n_ref;
  m, v, master   |x_gpu - x_ref| <= 1e-6 * max(|x_ref|, s), with s the operand
                 scale of the whole recurrence (the sum of the magnitudes of its
                 terms, so that cancellation in any step is covered):
                   m:      M_t = b1 M_{t-1} + (1 - b1) |gc_t|,           M_0 = 0
                   v:      |v_ref| (all terms are positive)
                   master: A_t = A_{t-1} (1 - lr wd) + lr |u_t|,           A_0 = |p_0|
                 with gc_t the clipped gradient and u_t = m_hat_t / (sqrt(v_hat_t) + eps)
                 of the oracle's step t;
  bf16 param     (a) bit-exact to the round-to-nearest-even bf16 of the GPU's own
                 FP32 master (checked with the oracle's pinned cast), and (b)
                 the RNE bf16 of some value within the master's tolerance of the
                 oracle's FP32 master: RNE is monotonic, so the GPU's bf16 must lie
                 in [RNE(p_ref - tol), RNE(p_ref + tol)].  Where tol is below half a
                 bf16 ulp this is "bit-exact except 1 ulp next to a rounding
                 midpoint"; for masters that cancel to far below their operand
                 scale it admits the few ulps their FP32 tolerance implies.
"""
import math
import os

import numpy as np
import torch

import oracle
import synth
from synth import gpu as sgpu
from mixed_precision_optimizer_bf16_gb300 import bf16opt as C
from mixed_precision_optimizer_bf16_gb300.optimizer import BF16Optimizer, alloc_flat

REL = 1e-6
SUBNORMAL_UNIT = 2.0 ** -149     # spacing of FP32 values below 2^-126


def ogroups(wl):
    """Oracle groups carry the FP32-rounded hyper-parameters the C ABI receives."""
    f = lambda x: float(np.float32(x))
    return [oracle.group(f(g["lr"]), f(g["beta1"]), f(g["beta2"]), f(g["eps"]), f(g["weight_decay"]))
            for g in wl.groups]


def _alloc(n, dtype, misalign, device="cuda"):
    base = torch.empty(n + misalign + 64, dtype=dtype, device=device)
    return base[misalign:misalign + n]


class GpuShard:
    """Device state of a workload + its bf16opt handle."""

    def __init__(self, wl, grad_scale=1.0, defer=False, grad_per_tensor=False):
        """defer: False, True (defer the last micro-batch only) or a per-micro-batch
        list of flags (deferred gradients then get buffers of their own).
        grad_per_tensor (LIST): every tensor's gradient gets a buffer of its
        own, offset like its state, instead of a slice of one flat buffer."""
        self.wl = wl
        G = wl.gas
        if defer is True:
            self.pattern = [False] * (G - 1) + [True]
        elif not defer:
            self.pattern = [False] * G
        else:
            self.pattern = [bool(x) for x in defer]
            assert len(self.pattern) == G
        self.defer = self.pattern[-1]
        self.norms = []
        # forced through the bulk-copy pipeline: the step must take it where its
        # stage fits (the accumulator with up to 2 pending gradients, or up to 4
        # without it) and the buffers are aligned alike (see expected_step_path)
        self.forced_pipe = os.environ.get("BF16OPT_PIPE") == "1"
        if wl.mode == "flat":
            self.flat = alloc_flat(wl.n, "cuda", wl.misalign)
            sgpu.fill_master(wl, self.flat["master"])
            for k in ("exp_avg", "exp_avg_sq", "grad_accum", "param_bf16"):
                self.flat[k].zero_()
            self.opt = BF16Optimizer(wl.groups, flat=self.flat, ranges=wl.ranges(), max_grad_norm=wl.max_norm,
                                     grad_scale=grad_scale)
        else:
            self.tensors = []
            master = _alloc(wl.n, torch.float32, 0)
            sgpu.fill_master(wl, master)
            for i, (t, off) in enumerate(zip(wl.tensors, wl.offsets)):
                d = dict(master=_alloc(t.numel, torch.float32, wl.misalign),
                         exp_avg=_alloc(t.numel, torch.float32, wl.misalign),
                         exp_avg_sq=_alloc(t.numel, torch.float32, wl.misalign),
                         grad_accum=_alloc(t.numel, torch.float32, wl.misalign),
                         param_bf16=_alloc(t.numel, torch.int16, wl.misalign), group=wl.group_of_tensor(i))
                d["master"].copy_(master[off:off + t.numel])
                for k in ("exp_avg", "exp_avg_sq", "grad_accum", "param_bf16"):
                    d[k].zero_()
                self.tensors.append(d)
            del master
            self.opt = BF16Optimizer(wl.groups, tensors=self.tensors, max_grad_norm=wl.max_norm,
                                     grad_scale=grad_scale)
        nbuf = wl.gas if any(self.pattern[:-1]) else 1
        self.gbufs = [_alloc(wl.n, torch.int16, wl.misalign) for _ in range(nbuf)]
        self.gbuf = self.gbufs[0]
        self.grad_per_tensor = bool(grad_per_tensor) and wl.mode != "flat"
        self.tgrads = ([[_alloc(t.numel, torch.int16, wl.misalign) for t in wl.tensors] for _ in range(nbuf)]
                       if self.grad_per_tensor else None)

    def grads_arg(self, buf=None):
        buf = self.gbuf if buf is None else buf
        if self.wl.mode == "flat":
            return buf
        return [buf[off:off + t.numel] for t, off in zip(self.wl.tensors, self.wl.offsets)]

    def run_step(self, step):
        wl = self.wl
        for k in range(wl.gas):
            buf = self.gbufs[k % len(self.gbufs)]
            sgpu.fill_grad(wl, step, k, buf)
            if self.grad_per_tensor:
                own = self.tgrads[k % len(self.gbufs)]
                for dst, t, off in zip(own, wl.tensors, wl.offsets):
                    dst.copy_(buf[off:off + t.numel])
                arg = own
            else:
                arg = self.grads_arg(buf)
            self.opt.accumulate(arg, first=(k == 0), last=(k == wl.gas - 1), defer=self.pattern[k])
        norm = self.opt.grad_norm(sync=True)
        self.opt.step()
        self.norms.append(norm)
        return norm

    def expected_step_path(self):
        """BF16OPT_PATH_* the fused step should have taken."""
        if self.wl.n == 0:
            return C.BF16OPT_PATH_NONE
        if not self.forced_pipe:
            return None
        pending = len(self.pattern) - max([k + 1 for k, d in enumerate(self.pattern) if not d], default=0)
        has_acc = not all(self.pattern)
        quad_bytes = (16 if has_acc else 0) + 8 * max(pending, 1) + 48
        # FLAT: every range's gradient starts at the range's own offset, as its
        # state does.  LIST: tensor i's gradient is a slice at offsets[i] of one
        # buffer while its state is allocated on its own, so the bf16 offsets
        # agree modulo 16 bytes only where offsets[i] is a multiple of 8.
        aligned = (self.wl.mode == "flat" or pending == 0 or self.grad_per_tensor or
                   all(off % 8 == 0 for t, off in zip(self.wl.tensors, self.wl.offsets) if t.numel))
        return C.BF16OPT_PATH_PIPELINE if quad_bytes <= 80 and aligned else C.BF16OPT_PATH_VECTOR

    def run(self, steps):
        for s in range(steps):
            self.run_step(s)
        torch.cuda.synchronize()
        want = self.expected_step_path()
        if want is not None and steps:
            assert C.bf16opt_step_path(self.opt.h) == (0, want), (C.bf16opt_step_path(self.opt.h), want)

    # ---- read back
    def full(self, name):
        if self.wl.mode == "flat":
            t = self.flat[name]
            return t.cpu().numpy()
        return np.concatenate([d[name].cpu().numpy() for d in self.tensors])

    def gather(self, name, idx):
        idx = np.asarray(idx, dtype=np.int64)
        if self.wl.mode == "flat":
            t = self.flat[name]
            return t[torch.from_numpy(idx).to(t.device)].cpu().numpy()
        tid = self.wl.tensor_of(idx)
        out = None
        for ti in np.unique(tid):
            sel = np.nonzero(tid == ti)[0]
            loc = idx[sel] - self.wl.offsets[ti]
            t = self.tensors[ti][name]
            vals = t[torch.from_numpy(loc).to(t.device)].cpu().numpy()
            if out is None:
                out = np.empty(idx.size, vals.dtype)
            out[sel] = vals
        return out

    def slice(self, name, lo, hi):
        """Elements [lo, hi) of one state buffer, copied to the host."""
        if self.wl.mode == "flat":
            return self.flat[name][lo:hi].cpu().numpy()
        parts = []
        for d, t, off in zip(self.tensors, self.wl.tensors, self.wl.offsets):
            a, b = max(lo, off), min(hi, off + t.numel)
            if a < b:
                parts.append(d[name][a - off:b - off].cpu().numpy())
        return np.concatenate(parts)

    def slice_states(self, lo, hi):
        get = lambda k: self.slice(k, lo, hi)
        return dict(p=get("master"), m=get("exp_avg"), v=get("exp_avg_sq"), acc=get("grad_accum"),
                    p_bf16=get("param_bf16").view(np.uint16))

    def acc_folded(self):
        """Micro-batches of the last step that the stored accumulator holds:
        up to the last micro-batch that was not deferred (0: never stored)."""
        return max([k + 1 for k, d in enumerate(self.pattern) if not d], default=0)

    def states(self, idx=None):
        get = (lambda k: self.full(k)) if idx is None else (lambda k: self.gather(k, idx))
        return dict(p=get("master"), m=get("exp_avg"), v=get("exp_avg_sq"), acc=get("grad_accum"),
                    p_bf16=get("param_bf16").view(np.uint16))

    def close(self):
        self.opt.close()


# ------------------------------------------------------------------ oracle side

def _gvec(wl, gof, attr):
    return np.array([getattr(g, attr) for g in ogroups(wl)])[gof]


def _update_scales(sc, wl, gof, acc, c, m, v, t, grad_scale):
    """Advance the operand scales M (first moment) and A (master) by one step."""
    b1, b2 = _gvec(wl, gof, "beta1"), _gvec(wl, gof, "beta2")
    lr, wd, eps = _gvec(wl, gof, "lr"), _gvec(wl, gof, "weight_decay"), _gvec(wl, gof, "eps")
    e = acc if grad_scale == 1.0 else (acc * np.float32(grad_scale)).astype(np.float32)
    gc = np.abs(e.astype(np.float64)) * c
    sc["M"] = b1 * sc["M"] + (1 - b1) * gc
    u = np.abs(m.astype(np.float64) / (1 - b1 ** t)) / (np.sqrt(v.astype(np.float64) / (1 - b2 ** t)) + eps)
    sc["A"] = sc["A"] * (1 - lr * wd) + lr * u


def oracle_dense(wl, steps, grad_scale=1.0):
    """Dense oracle run, one step at a time; returns (final states, operand scales)."""
    n = wl.n
    p = synth.fill_master(wl, np.empty(n, np.float32))
    G = ogroups(wl)
    gof = wl.group_of(np.arange(n))
    gfn = lambda s, k: synth.fill_grad(wl, s, k, np.empty(n, np.uint16))
    sc = {"M": np.zeros(n), "A": np.abs(p.astype(np.float64))}
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    sums, clips = [], []
    r = None
    for s in range(steps):
        r = oracle.run_dense(p, gfn, wl.ranges(), G, 1, wl.gas, wl.max_norm, grad_scale, t0=s, m=m, v=v)
        p, m, v = r["p"], r["m"], r["v"]
        sums += r["sumsq"]
        clips += r["clip"]
        _update_scales(sc, wl, gof, r["acc"], r["clip"][0], m, v, s + 1, grad_scale)
    r["sumsq"], r["clip"] = sums, clips
    return r, sc


def oracle_sampled(wl, steps, idx, grad_scale=1.0):
    """Streamed norms of every step + sampled whole-run replays."""
    st = oracle.stream(wl.id, wl.gas, synth.sigma_scale(wl.grad_sigma), synth.zero_thresh(wl.zero_frac),
                       grad_scale)
    sums = [oracle.stream_sumsq(st, s, wl.n) for s in range(steps)]
    clips = [oracle.clip_coef(S, wl.max_norm) for S in sums]
    idx = np.asarray(idx, dtype=np.uint64)
    p0 = synth.gather_master(wl, idx)
    G = ogroups(wl)
    gof = wl.group_of(idx)
    sc = {"M": np.zeros(idx.size), "A": np.abs(p0.astype(np.float64))}
    for s in range(steps):
        p, m, v, pb, acc = oracle.sample_run(st, idx, p0, G, gof, clips[:s + 1])
        _update_scales(sc, wl, gof, acc, clips[s], m, v, s + 1, grad_scale)
    fin = dict(p=p, m=m, v=v, p_bf16=pb, acc=acc, sumsq=sums, clip=clips)
    return fin, sc


def _oracle_slice(wl, lo, hi, steps, clips, snap_at, threads, grad_scale=1.0):
    """The oracle over elements [lo, hi) of a workload for `steps` steps with the
    given global clip coefficients (every element's arithmetic is its own; the
    norm is the only global quantity).  Returns (final states, operand scales,
    {k: the last step's accumulator after k micro-batches} for k in snap_at)."""
    S = hi - lo
    p = synth.fill_master(wl, np.empty(S, np.float32), lo, threads=threads)
    m, v = np.zeros(S, np.float32), np.zeros(S, np.float32)
    pb = oracle.f32_to_bf16(p, threads)
    G = ogroups(wl)
    gof = wl.group_of(np.arange(lo, hi, dtype=np.int64))
    rg = [(max(b, lo) - lo, min(e, hi) - lo, gi) for b, e, gi in wl.ranges() if max(b, lo) < min(e, hi)]
    sc = {"M": np.zeros(S), "A": np.abs(p.astype(np.float64))}
    acc, g = np.empty(S, np.float32), np.empty(S, np.uint16)
    snaps = {}
    for s in range(steps):
        for k in range(wl.gas):
            synth.fill_grad(wl, s, k, g, lo, threads=threads)
            oracle.accumulate(acc, g, first=k == 0, threads=threads)
            if s == steps - 1 and k + 1 in snap_at:
                snaps[k + 1] = acc.copy()
        for b, e, gi in rg:
            oracle.adamw(p[b:e], m[b:e], v[b:e], pb[b:e], acc[b:e], clips[s], G[gi], s + 1, grad_scale, threads)
        _update_scales(sc, wl, gof, acc, clips[s], m, v, s + 1, grad_scale)
    return dict(p=p, m=m, v=v, p_bf16=pb, acc=acc), sc, snaps


def dense_streamed_parity(wl, shards, steps, slice_elems=1 << 25, workers=4):
    """Every element of full-size shards against the oracle, one host slice at a time.

    shards: {name: GpuShard} that have run `steps` steps of `wl` (any deferral
    patterns).  The oracle's global sum of squares of every step is streamed
    from the generators' counters; then each slice of the shard is run through
    the oracle alone (inputs regenerated for the slice) and compared element by
    element with every shard's copy of that slice, the stored accumulator
    included wherever the shard stored one (bit-exact, after as many
    micro-batches as it folded).  Slices run `workers` at a time (numpy and the
    oracle release the GIL).  Returns ({name: merged stats}, per-step sums of squares)."""
    from concurrent.futures import ThreadPoolExecutor

    st = oracle.stream(wl.id, wl.gas, synth.sigma_scale(wl.grad_sigma), synth.zero_thresh(wl.zero_frac))
    sums = [oracle.stream_sumsq(st, s, wl.n) for s in range(steps)]
    clips = [oracle.clip_coef(S, wl.max_norm) for S in sums]
    folded = {name: sh.acc_folded() for name, sh in shards.items()}
    snap_at = {k for k in folded.values() if 0 < k < wl.gas}
    threads = max(1, oracle.nthreads() // workers)

    def one(lo):
        hi = min(wl.n, lo + slice_elems)
        ref, sc, snaps = _oracle_slice(wl, lo, hi, steps, clips, snap_at, threads)
        out = {}
        for name, sh in shards.items():
            k = folded[name]
            check = False if k == 0 else (True if k == wl.gas else snaps[k])
            out[name] = compare(sh.slice_states(lo, hi), ref, sc, wl, check_acc=check)
        return out

    with ThreadPoolExecutor(max_workers=workers) as ex:
        parts = list(ex.map(one, range(0, wl.n, slice_elems)))
    return {name: merge_stats([p[name] for p in parts]) for name in shards}, sums


def sample_indices(wl, k=1 << 15, seed=0):
    """Random elements plus every tensor's first/last element and chunk edges."""
    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, wl.n, size=min(k, wl.n), dtype=np.int64)]
    edges = []
    for t, off in zip(wl.tensors, wl.offsets):
        edges += [off, off + 1, off + t.numel - 1, off + t.numel - 2, off + min(t.numel - 1, 16383),
                  off + min(t.numel - 1, 16384)]
    edges += [0, wl.n - 1]
    idx.append(np.array([e for e in edges if 0 <= e < wl.n], np.int64))
    return np.unique(np.concatenate(idx))


# ------------------------------------------------------------------ comparison

def _bf16_interval(p_ref, scale):
    """[RNE(p_ref - tol), RNE(p_ref + tol)] as FP32 values, tol = REL * max(|p_ref|, scale),
    with the FP32 ends rounded outward."""
    x = p_ref.astype(np.float64)
    tol = REL * np.maximum(np.abs(x), scale)
    lo = (x - tol).astype(np.float32)
    lo = np.where(lo.astype(np.float64) > x - tol, np.nextafter(lo, np.float32(-np.inf)), lo)
    hi = (x + tol).astype(np.float32)
    hi = np.where(hi.astype(np.float64) < x + tol, np.nextafter(hi, np.float32(np.inf)), hi)
    return oracle.bf16_to_f32(oracle.f32_to_bf16(lo)), oracle.bf16_to_f32(oracle.f32_to_bf16(hi))


def _bf16_half_ulp(p_ref):
    """Half a bf16 unit in the last place at p_ref (FP64): bf16 keeps 8
    significant bits, so for 2^(e-1) <= |p| < 2^e the unit is 2^(e-8); below
    FP32's smallest normal value (2^-126) the spacing is fixed at 2^-133."""
    x = np.abs(p_ref.astype(np.float64))
    _, e = np.frexp(x)
    e = np.where(x == 0, -125, np.maximum(e, -125))
    return np.ldexp(1.0, e - 9)


def compare(gpu, ref, scales, wl, grad_scale=1.0, check_acc=True):
    """Element-wise parity; returns a stats dict, raises AssertionError on a breach.

    Elements whose FP32 bits equal the oracle's need no tolerance arithmetic;
    the bounds are evaluated on the others only (same outcome, less work on
    multi-GB shards)."""
    stats = {}
    if check_acc is not False:
        want = ref["acc"] if check_acc is True else check_acc
        bad = np.nonzero(gpu["acc"].view(np.uint32) != want.view(np.uint32))[0]
        # +0 and -0 compare equal
        bad = bad[~((gpu["acc"][bad] == 0) & (want[bad] == 0))]
        assert bad.size == 0, f"accumulator differs at {bad[:8]}: {gpu['acc'][bad[:8]]} vs {want[bad[:8]]}"
    # FP32's subnormal range has a fixed spacing of 2^-149, so a relative bound
    # cannot hold there: each step the two sides' roundings may land on
    # neighbouring subnormals, and earlier differences decay by beta < 1 per step,
    # so after T steps they differ by at most T units.
    floor = getattr(wl, "steps", 1) * SUBNORMAL_UNIT
    for name, skey in (("m", "M"), ("v", None), ("p", "A")):
        d = np.nonzero(gpu[name].view(np.uint32) != ref[name].view(np.uint32))[0]
        x, y = gpu[name][d].astype(np.float64), ref[name][d].astype(np.float64)
        s = np.abs(y) if skey is None else scales[skey][d]
        err = np.abs(x - y)
        lim = np.maximum(REL * np.maximum(np.abs(y), s), floor)
        bad = np.nonzero(~(err <= lim))[0]
        assert bad.size == 0, (f"{name} out of tolerance at {d[bad[:8]]}: gpu {x[bad[:8]]} ref {y[bad[:8]]} "
                               f"lim {lim[bad[:8]]}")
        stats[name + "_max_scaled_err"] = float(np.max(err / np.maximum(np.maximum(np.abs(y), s), 1e-45))) \
            if d.size else 0.0
        stats[name + "_strict_rel_fail"] = int(np.count_nonzero(err > REL * np.abs(y)))
        stats[name + "_bits_differ"] = int(d.size)
    # bf16 (a): the RNE cast of the GPU's own master, every element
    own = oracle.f32_to_bf16(gpu["p"])
    fin = ~np.isnan(gpu["p"])
    bad = np.nonzero(fin & (own != gpu["p_bf16"]))[0]
    assert bad.size == 0, f"bf16 is not the RNE cast of the GPU master at {bad[:8]}"
    # bf16 (b): where it differs from the oracle's, it must lie in
    # [RNE(p_ref - tol), RNE(p_ref + tol)] (RNE is monotonic, so an equal value does)
    d = np.nonzero(fin & (gpu["p_bf16"] != ref["p_bf16"]))[0]
    pr, A = ref["p"][d], scales["A"][d]
    lo, hi = _bf16_interval(pr, A)
    val = oracle.bf16_to_f32(gpu["p_bf16"][d])
    bad = np.nonzero(~((val >= lo) & (val <= hi)))[0]
    assert bad.size == 0, (f"bf16 params outside the master's tolerance at {d[bad[:8]]}: "
                           f"{gpu['p_bf16'][d[bad[:8]]]} vs {ref['p_bf16'][d[bad[:8]]]}")
    bg, br = gpu["p_bf16"][d].astype(np.int64), ref["p_bf16"][d].astype(np.int64)
    diff = np.abs(bg - br)
    diff[((bg & 0x7FFF) == 0) & ((br & 0x7FFF) == 0)] = 0
    # More than one bf16 unit apart is allowed only where the master's own FP32
    # tolerance is wider than half a bf16 unit at p_ref (a master that cancels
    # far below its operand scale); elsewhere the rule is "bit-exact, or one
    # unit next to a rounding midpoint".
    over = np.nonzero(diff > 1)[0]
    tol = REL * np.maximum(np.abs(pr[over].astype(np.float64)), A[over])
    unjust = np.nonzero(~(tol > _bf16_half_ulp(pr[over])))[0]
    assert unjust.size == 0, (f"bf16 more than one unit off where the master's tolerance is below half a bf16 "
                              f"unit, at {d[over[unjust[:8]]]}")
    stats["bf16_ulp_diffs"] = int(np.count_nonzero(diff))
    stats["bf16_max_ulp_diff"] = int(diff.max()) if diff.size else 0
    stats["bf16_diffs_over_1ulp"] = int(over.size)
    stats["elements"] = int(gpu["p"].size)
    return stats


def merge_stats(parts):
    """Combine compare() stats of disjoint slices."""
    out = {}
    for st in parts:
        for k, v in st.items():
            if k.endswith("_max_scaled_err") or k == "bf16_max_ulp_diff":
                out[k] = max(out.get(k, 0), v)
            else:
                out[k] = out.get(k, 0) + v
    return out


def check_norms(gpu_norms, ref_sums):
    for g, S in zip(gpu_norms, ref_sums):
        r = math.sqrt(S)
        assert abs(g - r) <= REL * r, f"norm {g} vs {r}"
    return max((abs(g - math.sqrt(S)) / math.sqrt(S) if S > 0 else abs(g)) for g, S in zip(gpu_norms, ref_sums))
