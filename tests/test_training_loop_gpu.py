"""The optimizer inside a real training loop.

A small bf16 model is trained with BF16Optimizer.from_parameters: autograd
writes each micro-batch's bf16 gradients into the optimizer's flat gradient
buffer (one reused buffer, or one per micro-batch), the library accumulates
them (the last micro-batch, or every one, deferred into the step), clips and
applies AdamW, and the model's parameters -- views into the flat bf16
parameter buffer -- change in place.  Every step is checked against
the oracle fed the very gradients autograd produced, with the parity tests'
tolerances, and the loss must fall.
"""
import math
from types import SimpleNamespace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import harness  # noqa: E402
import oracle  # noqa: E402
from harness import compare, ogroups  # noqa: E402
from mixed_precision_optimizer_bf16_gb300.optimizer import BF16Optimizer  # noqa: E402

pytestmark = pytest.mark.gpu


def _host(t, dtype):
    return t.detach().cpu().view(dtype).numpy().copy()


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
@pytest.mark.parametrize("resident", [False, True])
def test_training_loop_matches_oracle_every_step(resident):
    """resident=False: one gradient buffer, the last micro-batch deferred;
    resident=True: one gradient buffer per micro-batch and every micro-batch
    deferred (the accumulator is never stored)."""
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(48, 160), torch.nn.GELU(), torch.nn.Linear(160, 48))
    model = model.cuda().to(torch.bfloat16)
    decay = [p for name, p in model.named_parameters() if name.endswith("weight")]
    no_decay = [p for name, p in model.named_parameters() if name.endswith("bias")]
    gas = 3
    opt = BF16Optimizer.from_parameters([{"params": decay, "weight_decay": 0.01}, {"params": no_decay}],
                                        lr=1e-2, max_grad_norm=1.0, grad_buffers=gas if resident else 1)
    flat = opt.flat
    n = flat["master"].numel()
    base, end = flat["param_bf16"].data_ptr(), flat["param_bf16"].data_ptr() + 2 * n
    assert all(base <= p.data_ptr() < end for p in model.parameters())      # parameters live in the shard

    ns = SimpleNamespace(groups=opt.groups)
    G = ogroups(ns)
    gof = np.zeros(n, np.int64)
    for b, e, gi in opt.ranges:
        gof[b:e] = gi
    p = _host(flat["master"], torch.float32)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    sc = {"M": np.zeros(n), "A": np.abs(p.astype(np.float64))}

    gen = torch.Generator(device="cuda").manual_seed(1)
    losses = []
    for step in range(5):
        grads = []
        for k in range(gas):
            if resident:
                opt.use_grad_buffer(k)
            else:
                opt.zero_grad()
            x = torch.randn(64, 48, device="cuda", generator=gen).to(torch.bfloat16)
            y = 0.5 * torch.roll(x, 1, dims=1)
            loss = ((model(x).float() - y.float()) ** 2).mean()
            loss.backward()
            grads.append(_host(opt.grad_buffer, torch.int16).view(np.uint16))
            opt.accumulate(first=k == 0, last=k == gas - 1, defer=resident or k == gas - 1)
            losses.append(loss.item())
        norm = opt.grad_norm(sync=True)
        opt.step()
        torch.cuda.synchronize()

        ref = oracle.run_dense(p, lambda s, kk: grads[kk], opt.ranges, G, 1, gas, 1.0, t0=step, m=m, v=v)
        p, m, v = ref["p"], ref["m"], ref["v"]
        harness._update_scales(sc, ns, gof, ref["acc"], ref["clip"][0], m, v, step + 1, 1.0)
        S = ref["sumsq"][0]
        assert abs(norm - math.sqrt(S)) <= harness.REL * math.sqrt(S)
        got = dict(p=_host(flat["master"], torch.float32), m=_host(flat["exp_avg"], torch.float32),
                   v=_host(flat["exp_avg_sq"], torch.float32),
                   p_bf16=_host(flat["param_bf16"], torch.int16).view(np.uint16))
        compare(got, ref, sc, ns, check_acc=False)
    assert np.mean(losses[-gas:]) < np.mean(losses[:gas])
    opt.close()
