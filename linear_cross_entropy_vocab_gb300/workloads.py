"""Seeded synthetic inputs for fused linear cross-entropy workloads.

This module only draws random tensors. It holds none of the loss arithmetic, so
both the CUDA path and the fp64 oracle can be fed from it without sharing any
of the method's computation.

Workload shapes follow the Llama-3 LM-head shape (H=4096, V=128256) and the
32000-vocabulary shapes that the fused-linear-loss pull requests benchmark
(Liger-Kernel PR #1423 "Benchmark" tables; Liger-Kernel PR #1287
"Benchmarks"), plus a softcapped head and a long batch.

Readings of the workload notation (stated once, used everywhere):
  * ``N(0, x)`` gives the variance ``x`` (so ``N(0, 1/H)`` has std ``H**-0.5``
    and ``N(0, 2)`` has std ``sqrt(2)``).
  * Zipf(s) over V: P(rank k) proportional to ``k**-s`` for ``k = 1..V`` and
    token id ``k - 1``, sampled by inverting the fp64 CDF with uniform draws.
  * An ignore fraction ``f`` marks exactly ``round(f * N)`` rows, chosen by a
    seeded permutation, with ``ignore_index``.
  * "1% of weight rows scaled x8": ``round(0.01 * V)`` rows chosen by a seeded
    permutation are multiplied by 8 after sampling and before the bf16 cast.
  * Draw order: hidden, weight, bias, ignore permutation, targets, scaled
    rows, then (KL divergence only) teacher logits as draw 6; draw ``idx``
    uses ``torch.Generator('cpu').manual_seed(seed + idx)``.
    Values are drawn in fp32 and cast to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "make_teacher_probs", "peaked_rows",
           "gemm_flops"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n: int
    h: int
    v: int
    dtype: str  # "f32", "bf16" or "f16"
    hidden_var: float = 1.0
    weight_var: Optional[float] = None  # None: 1/H
    bias_var: Optional[float] = None  # None: no bias
    targets: str = "uniform"  # "uniform" or "zipf"
    zipf_s: float = 1.1
    ignore_frac: float = 0.0
    ignore_index: int = -100
    logit_scale: float = 1.0
    softcap: Optional[float] = None
    reduction: str = "mean"
    return_metrics: bool = False
    peaked_frac: float = 0.0
    peaked_factor: float = 8.0
    seed: int = 0
    label_smoothing: float = 0.0
    z_loss: float = 0.0

    def with_shape(self, n: Optional[int] = None, h: Optional[int] = None,
                   v: Optional[int] = None, **kw) -> "Workload":
        """Same value recipe at another shape (tail and small-case variants)."""
        return dataclasses.replace(self, n=self.n if n is None else n,
                                   h=self.h if h is None else h,
                                   v=self.v if v is None else v, **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[self.dtype]


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fp32", 256, 128, 1000, "f32", ignore_frac=0.05,
                 return_metrics=True),
        Workload("mid_bf16", 4096, 2048, 32000, "bf16", bias_var=0.02,
                 targets="zipf", ignore_frac=0.10),
        Workload("llama3_head_bf16", 8192, 4096, 128256, "bf16",
                 ignore_frac=0.02, return_metrics=True),
        Workload("softcap_bf16", 16384, 3584, 152064, "bf16", hidden_var=2.0,
                 ignore_frac=0.30, logit_scale=0.5, softcap=30.0,
                 reduction="sum"),
        Workload("long_bf16", 32768, 4096, 128256, "bf16", ignore_frac=0.05,
                 peaked_frac=0.01, reduction="mean"),
    ]
}


def _gen(seed: int, idx: int) -> torch.Generator:
    return torch.Generator("cpu").manual_seed(seed + idx)


def make_inputs(w: Workload) -> dict:
    """Draw hidden [N,H], weight [V,H], bias [V] or None, targets int64 [N] on
    the CPU, in the workload's dtype (targets always int64)."""
    n, h, v = w.n, w.h, w.v
    hidden = torch.randn(n, h, generator=_gen(w.seed, 0), dtype=torch.float32)
    hidden.mul_(math.sqrt(w.hidden_var))
    wvar = (1.0 / h) if w.weight_var is None else w.weight_var
    weight = torch.randn(v, h, generator=_gen(w.seed, 1), dtype=torch.float32)
    weight.mul_(math.sqrt(wvar))
    bias = None
    if w.bias_var is not None:
        bias = torch.randn(v, generator=_gen(w.seed, 2), dtype=torch.float32)
        bias.mul_(math.sqrt(w.bias_var))
    n_ignore = int(round(w.ignore_frac * n))
    ignore_rows = torch.randperm(n, generator=_gen(w.seed, 3))[:n_ignore]
    g_t = _gen(w.seed, 4)
    if w.targets == "uniform":
        targets = torch.randint(0, v, (n,), generator=g_t, dtype=torch.int64)
    elif w.targets == "zipf":
        k = torch.arange(1, v + 1, dtype=torch.float64)
        cdf = torch.cumsum(k.pow(-w.zipf_s), 0)
        cdf /= cdf[-1].clone()
        u = torch.rand(n, generator=g_t, dtype=torch.float64)
        targets = torch.searchsorted(cdf, u).clamp_(max=v - 1).to(torch.int64)
    else:
        raise ValueError(f"unknown target distribution {w.targets!r}")
    targets[ignore_rows] = w.ignore_index
    if w.peaked_frac > 0:
        n_peak = int(round(w.peaked_frac * v))
        rows = torch.randperm(v, generator=_gen(w.seed, 5))[:n_peak]
        weight[rows] *= w.peaked_factor
    dt = w.torch_dtype
    return {
        "hidden": hidden.to(dt),
        "weight": weight.to(dt),
        "bias": None if bias is None else bias.to(dt),
        "targets": targets,
    }


def make_teacher_probs(w: Workload, teacher_std: float = 2.0, keep_top: Optional[int] = None,
                       idx: int = 6) -> torch.Tensor:
    """Teacher probabilities [N,V] for the KL divergence, in the workload's
    dtype: the distribution a teacher model would output, drawn as the
    softmax (fp32) of N(0, teacher_std**2) teacher logits (draw ``idx``).
    With ``keep_top`` k, each row keeps only its k largest entries
    (renormalised; the rest exactly 0), as a top-k truncated teacher does.
    These are inputs of the method; after the cast a row sums to 1 only up
    to the dtype's rounding."""
    t = torch.randn(w.n, w.v, generator=_gen(w.seed, idx), dtype=torch.float32)
    t.mul_(teacher_std)
    if keep_top is not None and keep_top < w.v:
        kth = torch.topk(t, keep_top, dim=1).values[:, -1:]
        t = t.masked_fill(t < kth, float("-inf"))
    q = torch.softmax(t, dim=1)
    return q.to(w.torch_dtype)


def peaked_rows(w: Workload) -> torch.Tensor:
    """The weight rows that make_inputs scaled by ``peaked_factor`` (same draw)."""
    if w.peaked_frac <= 0:
        return torch.empty(0, dtype=torch.int64)
    n_peak = int(round(w.peaked_frac * w.v))
    return torch.randperm(w.v, generator=_gen(w.seed, 5))[:n_peak]


def gemm_flops(n: int, h: int, v: int) -> float:
    """Algorithmic FLOPs of one forward+backward: four N x H x V contractions
    (forward logits, backward recompute, grad_hidden, grad_weight)."""
    return 8.0 * n * h * v
