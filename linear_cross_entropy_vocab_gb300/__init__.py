"""Fused linear cross-entropy for one GB300 GPU (sm_103a).

``fused_linear_cross_entropy`` computes the cross-entropy of
``softcap(logit_scale * (hidden @ weight.T + bias))`` against ``targets``
without materialising the (N, V) logits, with the metrics and gradients of
the "fused-linear-ce" model card (trl-lib). The compute runs in the
hand-written CUDA kernels of ``libflce.so`` (C ABI: include/flce.h); this
package marshals tensors to it.
"""
from .api import fused_linear_cross_entropy, flce_backward_tensors, flce_forward_tensors  # noqa: F401
from .native_build import build  # noqa: F401

__all__ = ["fused_linear_cross_entropy", "flce_forward_tensors", "flce_backward_tensors",
           "build"]
