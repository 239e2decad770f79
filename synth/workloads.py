"""The five optimizer-step workloads, as tensor tables (shapes, groups, init).

Sources for shapes and hyper-parameters:
  * "单机多卡实战：Megatron-DeepSpeed训练类BLOOM模型全流程解析", section 2 (model
    table: hidden 2048, 24 layers, 16 heads, vocab 250880) and section 3 (lr 6e-5,
    weight_decay 0.01, clip_grad 1.0, gradient_accumulation_steps 4);
  * "Как обучали BLOOM ...", section on Megatron tensor parallelism (hidden 14336);
  * "企业官网建设流程全解析" (cf-1.com), section 2.2 (GAS 32) and 3.3 (AdamW config).
Betas (0.9, 0.95) and eps 1e-8 are not on the pages; they come from the
workload definitions.  All inputs are seeded and synthetic: no dataset, token
or trained weight is used.

Init rules (plainest reading): weight matrices and embeddings ~N(0, 0.02),
LayerNorm gamma = 1, LayerNorm beta and biases = 0, m = v = 0.  LayerNorm and
bias tensors form the no-decay group (weight_decay 0).
"""
from dataclasses import dataclass, field

import numpy as np

LR, BETA1, BETA2, EPS, WD = 6e-5, 0.9, 0.95, 1e-8, 0.01
MAX_NORM = 1.0


@dataclass
class Tensor:
    name: str
    numel: int
    decay: bool
    init: tuple  # ("normal", sigma) | ("const", value) | ("loguniform", e_lo, e_hi)
    group: int = -1  # parameter group; -1: 0 if it decays, else 1


@dataclass
class Workload:
    id: int
    name: str
    tensors: list
    mode: str            # "flat": one contiguous buffer; "list": one allocation per tensor
    gas: int
    steps: int
    grad_sigma: float
    zero_frac: float = 0.0
    misalign: int = 0    # every device buffer starts this many elements past a 256-B boundary
    max_norm: float = MAX_NORM
    groups: list = field(default_factory=lambda: [
        dict(lr=LR, beta1=BETA1, beta2=BETA2, eps=EPS, weight_decay=WD),
        dict(lr=LR, beta1=BETA1, beta2=BETA2, eps=EPS, weight_decay=0.0)])

    def __post_init__(self):
        self.offsets = np.cumsum([0] + [t.numel for t in self.tensors[:-1]]).astype(np.int64).tolist()
        self.n = int(sum(t.numel for t in self.tensors))
        self._ends = np.array([o + t.numel for o, t in zip(self.offsets, self.tensors)], dtype=np.int64)

    def group_of_tensor(self, i):
        t = self.tensors[i]
        return t.group if t.group >= 0 else (0 if t.decay else 1)

    def tensor_of(self, idx):
        """Tensor index of each global element index."""
        return np.searchsorted(self._ends, np.asarray(idx, dtype=np.int64), side="right")

    def group_of(self, idx):
        grp = np.array([self.group_of_tensor(i) for i in range(len(self.tensors))], dtype=np.uint32)
        return grp[self.tensor_of(idx)]

    def ranges(self):
        """Flat-mode group ranges [begin, end, group], neighbours of one group merged."""
        out = []
        for i, (t, off) in enumerate(zip(self.tensors, self.offsets)):
            g = self.group_of_tensor(i)
            if out and out[-1][2] == g and out[-1][1] == off:
                out[-1][1] = off + t.numel
            else:
                out.append([off, off + t.numel, g])
        return out

    def bytes_per_step(self, deferred=False):
        """Algorithmic HBM bytes of one full step (accumulate x GAS, norm fused, step)."""
        g = self.gas
        if deferred:
            return self.n * ((6 if g > 1 else 0) + 10 * max(g - 2, 0) + (6 if g > 1 else 2) + 30 + 2)
        return self.n * (6 + 10 * (g - 1) + 30)


def _bloom_scaled():
    """Scaled-down BLOOM: hidden 2048, 24 layers, vocab 250880, tied embeddings."""
    h, L, V = 2048, 24, 250880
    w = ("normal", 0.02)
    one, zero = ("const", 1.0), ("const", 0.0)
    ts = [Tensor("word_embeddings", V * h, True, w),
          Tensor("emb_ln.gamma", h, False, one), Tensor("emb_ln.beta", h, False, zero)]
    for l in range(L):
        p = f"h.{l}."
        ts += [Tensor(p + "ln1.gamma", h, False, one), Tensor(p + "ln1.beta", h, False, zero),
               Tensor(p + "qkv.weight", 3 * h * h, True, w), Tensor(p + "qkv.bias", 3 * h, False, zero),
               Tensor(p + "proj.weight", h * h, True, w), Tensor(p + "proj.bias", h, False, zero),
               Tensor(p + "ln2.gamma", h, False, one), Tensor(p + "ln2.beta", h, False, zero),
               Tensor(p + "fc1.weight", 4 * h * h, True, w), Tensor(p + "fc1.bias", 4 * h, False, zero),
               Tensor(p + "fc2.weight", 4 * h * h, True, w), Tensor(p + "fc2.bias", h, False, zero)]
    ts += [Tensor("ln_f.gamma", h, False, one), Tensor("ln_f.beta", h, False, zero)]
    return ts


def _bloom176_tp4_slice(layers=6):
    """One TP=4 slice of BLOOM-176B layers (hidden 14336), one allocation per tensor."""
    h, tp = 14336, 4
    w = ("normal", 0.02)
    one, zero = ("const", 1.0), ("const", 0.0)
    ts = []
    for l in range(layers):
        p = f"h.{l}."
        ts += [Tensor(p + "ln1.gamma", h, False, one), Tensor(p + "ln1.beta", h, False, zero),
               Tensor(p + "qkv.weight", (3 * h // tp) * h, True, w), Tensor(p + "qkv.bias", h, False, zero),
               Tensor(p + "proj.weight", h * (h // tp), True, w), Tensor(p + "proj.bias", h, False, zero),
               Tensor(p + "ln2.gamma", h, False, one), Tensor(p + "ln2.beta", h, False, zero),
               Tensor(p + "fc1.weight", (4 * h // tp) * h, True, w), Tensor(p + "fc1.bias", h, False, zero),
               Tensor(p + "fc2.weight", h * (4 * h // tp), True, w), Tensor(p + "fc2.bias", h, False, zero)]
    return ts


def _make():
    return {
        1: Workload(1, "tiny flat shard 1,048,576", [Tensor("flat", 1 << 20, True, ("normal", 0.02))],
                    "flat", gas=4, steps=3, grad_sigma=1e-3),
        2: Workload(2, "scaled-down BLOOM 1.72B flat (hidden 2048, 24 layers, vocab 250880)", _bloom_scaled(),
                    "flat", gas=4, steps=2, grad_sigma=1e-4),
        3: Workload(3, "large ZeRO partition 1.83e9 flat", [Tensor("flat", 1_830_000_000, True, ("normal", 0.02))],
                    "flat", gas=32, steps=1, grad_sigma=5e-5),
        4: Workload(4, "ragged TP=4 slice of 6 BLOOM-176B layers (72 tensors)", _bloom176_tp4_slice(),
                    "list", gas=8, steps=2, grad_sigma=1e-4),
        5: Workload(5, "clipping edge 2^27+13, misaligned by 2",
                    [Tensor("flat", (1 << 27) + 13, True, ("loguniform", -26, 9))],
                    "flat", gas=2, steps=5, grad_sigma=0.01, zero_frac=0.01, misalign=2),
    }


WORKLOADS = _make()


def workload(i):
    return WORKLOADS[i]


def prefix(wl, n):
    """The first n elements of a flat workload (tensors cut at n), same ids and streams."""
    ts, left = [], n
    for t in wl.tensors:
        if left <= 0:
            break
        k = min(t.numel, left)
        ts.append(Tensor(t.name, k, t.decay, t.init))
        left -= k
    w = Workload(wl.id, f"{wl.name}, first {n} elements", ts, wl.mode, gas=wl.gas, steps=wl.steps,
                 grad_sigma=wl.grad_sigma, zero_frac=wl.zero_frac, misalign=wl.misalign, max_norm=wl.max_norm)
    w.groups = [dict(g) for g in wl.groups]
    return w


def custom(wl_id, sizes, decay=None, gas=2, steps=2, grad_sigma=1e-3, misalign=0, zero_frac=0.0,
           mode="flat", init=("normal", 0.02), max_norm=MAX_NORM):
    """Small ad-hoc workload for parity cases (ragged sizes, misalignment, GAS)."""
    decay = decay if decay is not None else [True] * len(sizes)
    ts = [Tensor(f"t{i}", int(n), bool(d), init) for i, (n, d) in enumerate(zip(sizes, decay))]
    return Workload(wl_id, f"custom {list(sizes)}", ts, mode, gas=gas, steps=steps, grad_sigma=grad_sigma,
                    zero_frac=zero_frac, misalign=misalign, max_norm=max_norm)
