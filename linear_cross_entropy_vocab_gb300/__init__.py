"""Fused linear cross-entropy for one GB300 GPU (sm_103a).

``fused_linear_cross_entropy`` computes the cross-entropy of
``softcap(logit_scale * (hidden @ weight.T + bias))`` against ``targets``
without materialising the (N, V) logits, with the metrics and gradients of
the "fused-linear-ce" model card (trl-lib). The compute runs in the
hand-written CUDA kernels of ``libflce.so`` (C ABI: include/flce.h); this
package marshals tensors to it. ``fused_linear_kl_div`` is the same fused
projection with a KL divergence against teacher probabilities
(FusedLinearKLDivLoss pull request, Liger-Kernel #1423).
"""
from .api import (  # noqa: F401
    flce_backward_tensors, flce_forward_tensors, flce_kl_backward_tensors,
    flce_kl_forward_tensors, fused_linear_cross_entropy, fused_linear_kl_div)
from .native_build import build  # noqa: F401

__all__ = ["fused_linear_cross_entropy", "flce_forward_tensors", "flce_backward_tensors",
           "fused_linear_kl_div", "flce_kl_forward_tensors", "flce_kl_backward_tensors",
           "build"]
