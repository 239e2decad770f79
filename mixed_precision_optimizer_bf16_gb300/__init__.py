"""BF16 mixed-precision optimizer step for one GB300 GPU (sm_103a).

FP32 accumulation of bf16 micro-batch gradients, deterministic global-norm
clipping and fused AdamW + bf16 cast over a rank's flat or ragged parameter
shard, behind the C ABI of include/bf16opt.h.  `bf16opt` is the Python
binding (same names); `optimizer.BF16Optimizer` drives it from torch tensors.
"""
from . import bf16opt  # noqa: F401
