"""Tensor-level API over the C ABI.

``fused_linear_cross_entropy`` has the signature of the "fused-linear-ce"
model card (trl-lib), §Full signature:

    fused_linear_cross_entropy(hidden (N,H), weight (V,H), targets (N,) int64,
        bias=None, ignore_index=-100, logit_scale=1.0, softcap=None,
        reduction="mean", return_metrics=False)
      -> loss | (loss, {"mean_token_accuracy": ..., "entropy": ...})

hidden, weight and bias receive gradients; the metrics are forward-only
(§Metrics for free). PyTorch supplies device memory and the current stream;
every step of the computation runs in libflce.so's kernels.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import abi

__all__ = ["fused_linear_cross_entropy", "flce_forward_tensors", "flce_backward_tensors",
           "fused_linear_kl_div", "flce_kl_forward_tensors", "flce_kl_backward_tensors"]


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return abi.FLCE_F32
    if t.dtype == torch.bfloat16:
        return abi.FLCE_BF16
    if t.dtype == torch.float16:
        return abi.FLCE_F16
    raise TypeError(f"unsupported dtype {t.dtype}: use float32, bfloat16 or float16")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _check_inputs(hidden, weight, targets, bias):
    if hidden.dim() != 2 or weight.dim() != 2 or hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden must be (N, H) and weight (V, H)")
    if targets.dim() != 1 or targets.shape[0] != hidden.shape[0]:
        raise ValueError("targets must be (N,)")
    if targets.dtype != torch.int64:
        raise TypeError("targets must be int64")
    if weight.dtype != hidden.dtype or (bias is not None and bias.dtype != hidden.dtype):
        raise TypeError("hidden, weight and bias must share one dtype")
    if bias is not None and (bias.dim() != 1 or bias.shape[0] != weight.shape[0]):
        raise ValueError("bias must be (V,)")
    for name, t in (("hidden", hidden), ("weight", weight), ("targets", targets), ("bias", bias)):
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device != hidden.device:
            raise ValueError(f"{name} is on {t.device}, hidden on {hidden.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


def flce_forward_tensors(hidden, weight, targets, bias=None, ignore_index=-100,
                         logit_scale=1.0, softcap=None, reduction="mean",
                         return_metrics=False, row_metrics=False, err_word=None,
                         vocab_chunk=0, skip_ignored=False, label_smoothing=0.0,
                         z_loss=0.0) -> dict:
    """Run flce_forward; returns a dict of freshly allocated output tensors:
    loss (0-d, or [N] for 'none'), loss_rows, lse_rows, n_valid (0-d int32),
    metrics ([2] or None), correct_rows / entropy_rows (when row_metrics).
    ``skip_ignored`` leaves ignored rows out of the contractions (their
    lse_rows / entropy_rows are then NaN)."""
    _check_inputs(hidden, weight, targets, bias)
    n, h = hidden.shape
    v = weight.shape[0]
    dev = hidden.device
    prob = abi.make_problem(n, h, v, _dtype_code(hidden), bias is not None, ignore_index,
                            logit_scale, softcap, reduction, vocab_chunk=vocab_chunk,
                            skip_ignored=skip_ignored, label_smoothing=label_smoothing,
                            z_loss=z_loss)
    f32 = dict(dtype=torch.float32, device=dev)
    loss_rows = torch.empty(n, **f32)
    lse_rows = torch.empty(n, **f32)
    n_valid = torch.empty((), dtype=torch.int32, device=dev)
    loss_out = None if reduction == "none" else torch.empty((), **f32)
    metrics = torch.empty(2, **f32) if return_metrics else None
    correct_rows = torch.empty(n, dtype=torch.int32, device=dev) if row_metrics else None
    entropy_rows = torch.empty(n, **f32) if row_metrics else None
    with torch.cuda.device(dev):
        ws_bytes = abi.flce_forward_workspace_size(prob)
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev).cuda_stream
        abi.flce_forward(prob, _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets),
                         _ptr(loss_rows), _ptr(lse_rows), _ptr(correct_rows),
                         _ptr(entropy_rows), _ptr(loss_out), _ptr(metrics), _ptr(n_valid),
                         _ptr(err_word), _ptr(ws), ws_bytes, stream)
    return {
        "loss": loss_rows if reduction == "none" else loss_out,
        "loss_rows": loss_rows,
        "lse_rows": lse_rows,
        "n_valid": n_valid,
        "metrics": metrics,
        "correct_rows": correct_rows,
        "entropy_rows": entropy_rows,
    }


def flce_backward_tensors(hidden, weight, targets, lse_rows, n_valid, grad_out, bias=None,
                          ignore_index=-100, logit_scale=1.0, softcap=None,
                          reduction="mean", grad_weight_dtype=None, err_word=None,
                          vocab_chunk=0, skip_ignored=False, label_smoothing=0.0,
                          z_loss=0.0):
    """Run flce_backward; returns (grad_hidden, grad_weight, grad_bias).
    ``grad_out`` is a 0-d fp32 tensor ('sum'/'mean') or [N] ('none').
    ``grad_weight_dtype`` torch.float32 keeps grad_weight in fp32.
    ``skip_ignored`` leaves ignored rows out of the contractions."""
    _check_inputs(hidden, weight, targets, bias)
    n, h = hidden.shape
    v = weight.shape[0]
    dev = hidden.device
    gw_dtype = hidden.dtype if grad_weight_dtype is None else grad_weight_dtype
    gw_code = abi.FLCE_F32 if gw_dtype == torch.float32 else _dtype_code(hidden)
    prob = abi.make_problem(n, h, v, _dtype_code(hidden), bias is not None, ignore_index,
                            logit_scale, softcap, reduction, grad_weight_dtype=gw_code,
                            vocab_chunk=vocab_chunk, skip_ignored=skip_ignored,
                            label_smoothing=label_smoothing, z_loss=z_loss)
    grad_out = grad_out.to(device=dev, dtype=torch.float32).contiguous()
    grad_hidden = torch.empty_like(hidden)
    grad_weight = torch.empty(v, h, dtype=gw_dtype, device=dev)
    grad_bias = torch.empty_like(bias) if bias is not None else None
    with torch.cuda.device(dev):
        ws_bytes = abi.flce_backward_workspace_size(prob)
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev).cuda_stream
        abi.flce_backward(prob, _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets),
                          _ptr(lse_rows), _ptr(n_valid), _ptr(grad_out), _ptr(grad_hidden),
                          _ptr(grad_weight), _ptr(grad_bias), _ptr(err_word), _ptr(ws),
                          ws_bytes, stream)
    return grad_hidden, grad_weight, grad_bias


class _FusedLinearCrossEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, weight, bias, targets, ignore_index, logit_scale, softcap,
                reduction, return_metrics, label_smoothing, z_loss, vocab_chunk):
        # ignored rows contribute nothing, so they are left out of the GEMMs
        out = flce_forward_tensors(hidden, weight, targets, bias, ignore_index, logit_scale,
                                   softcap, reduction, return_metrics, skip_ignored=True,
                                   label_smoothing=label_smoothing, z_loss=z_loss)
        ctx.save_for_backward(hidden, weight, bias, targets, out["lse_rows"], out["n_valid"])
        ctx.opts = (ignore_index, logit_scale, softcap, reduction, label_smoothing, z_loss,
                    vocab_chunk)
        metrics = out["metrics"]
        if metrics is None:
            metrics = torch.empty(0, dtype=torch.float32, device=hidden.device)
        ctx.mark_non_differentiable(metrics)
        return out["loss"], metrics

    @staticmethod
    def backward(ctx, grad_loss, _grad_metrics):
        hidden, weight, bias, targets, lse_rows, n_valid = ctx.saved_tensors
        (ignore_index, logit_scale, softcap, reduction, label_smoothing, z_loss,
         vocab_chunk) = ctx.opts
        gh, gw, gb = flce_backward_tensors(hidden, weight, targets, lse_rows, n_valid,
                                           grad_loss, bias, ignore_index, logit_scale,
                                           softcap, reduction, skip_ignored=True,
                                           label_smoothing=label_smoothing, z_loss=z_loss,
                                           vocab_chunk=vocab_chunk)
        need = ctx.needs_input_grad
        return (gh if need[0] else None, gw if need[1] else None,
                gb if (bias is not None and need[2]) else None,
                None, None, None, None, None, None, None, None, None)


def fused_linear_cross_entropy(hidden: torch.Tensor, weight: torch.Tensor,
                               targets: torch.Tensor, bias: Optional[torch.Tensor] = None,
                               ignore_index: int = -100, logit_scale: float = 1.0,
                               softcap: Optional[float] = None, reduction: str = "mean",
                               return_metrics: bool = False, *,
                               label_smoothing: float = 0.0, z_loss: float = 0.0,
                               vocab_chunk: int = 0):
    """Cross-entropy of softcap(logit_scale * (hidden @ weight.T + bias))
    against targets, without materialising the (N, V) logits. hidden may
    carry leading batch dimensions ([..., H] with targets [...]); its rows
    are flattened.

    Returns the loss (0-d for 'mean'/'sum', targets-shaped for 'none'), or with
    return_metrics ``(loss, {"mean_token_accuracy": 0-d, "entropy": 0-d})``;
    metrics are over non-ignored positions, entropy in nats.

    Keyword-only extras: ``label_smoothing`` eps (cross-entropy against
    (1-eps)*onehot + eps/V) and ``z_loss`` lam (adds lam * lse^2 per row).
    ``vocab_chunk`` bounds the vocabulary columns of the backward's dlogits
    buffer (rounded up to a multiple of 256); 0 takes the library's default
    (about a fifth of the vocabulary and at most a 512 MiB buffer). A
    smaller chunk lowers peak memory at some cost in speed.
    """
    if reduction not in abi.REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(abi.REDUCTIONS)}")
    batch_shape = targets.shape
    if hidden.dim() > 2:  # leading batch dimensions: rows are flattened
        if hidden.shape[:-1] != targets.shape:
            raise ValueError("hidden [..., H] and targets [...] must share the leading shape")
        hidden = hidden.reshape(-1, hidden.shape[-1])
        targets = targets.reshape(-1)
    hidden = hidden.contiguous()
    weight = weight.contiguous()
    targets = targets.contiguous()
    bias = None if bias is None else bias.contiguous()
    loss, metrics = _FusedLinearCrossEntropy.apply(hidden, weight, bias, targets,
                                                   int(ignore_index), float(logit_scale),
                                                   softcap, reduction, bool(return_metrics),
                                                   float(label_smoothing), float(z_loss),
                                                   int(vocab_chunk))
    if reduction == "none":
        loss = loss.reshape(batch_shape)
    if not return_metrics:
        return loss
    return loss, {"mean_token_accuracy": metrics[0], "entropy": metrics[1]}


# ------------------------------------------------------------ KL divergence
def _check_kl_inputs(hidden, weight, target_probs, labels, bias):
    if hidden.dim() != 2 or weight.dim() != 2 or hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden must be (N, H) and weight (V, H)")
    if target_probs.shape != (hidden.shape[0], weight.shape[0]):
        raise ValueError("target_probs must be (N, V)")
    if labels is not None:
        if labels.dim() != 1 or labels.shape[0] != hidden.shape[0]:
            raise ValueError("labels must be (N,)")
        if labels.dtype != torch.int64:
            raise TypeError("labels must be int64")
    if (weight.dtype != hidden.dtype or target_probs.dtype != hidden.dtype
            or (bias is not None and bias.dtype != hidden.dtype)):
        raise TypeError("hidden, weight, target_probs and bias must share one dtype")
    if bias is not None and (bias.dim() != 1 or bias.shape[0] != weight.shape[0]):
        raise ValueError("bias must be (V,)")
    for name, t in (("hidden", hidden), ("weight", weight), ("target_probs", target_probs),
                    ("labels", labels), ("bias", bias)):
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device != hidden.device:
            raise ValueError(f"{name} is on {t.device}, hidden on {hidden.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


def flce_kl_forward_tensors(hidden, weight, target_probs, labels=None, bias=None,
                            ignore_index=-100, temperature=1.0, eps=1e-10,
                            reduction="batchmean", err_word=None, skip_ignored=False) -> dict:
    """Run flce_kl_forward; returns loss (0-d, or [N] for 'none'), loss_rows,
    lse_rows, qsum_rows and n_counted (0-d int32)."""
    _check_kl_inputs(hidden, weight, target_probs, labels, bias)
    n, h = hidden.shape
    v = weight.shape[0]
    dev = hidden.device
    prob = abi.make_kl_problem(n, h, v, _dtype_code(hidden), bias is not None, ignore_index,
                               temperature, eps, reduction, skip_ignored=skip_ignored)
    f32 = dict(dtype=torch.float32, device=dev)
    loss_rows = torch.empty(n, **f32)
    lse_rows = torch.empty(n, **f32)
    qsum_rows = torch.empty(n, **f32)
    n_counted = torch.empty((), dtype=torch.int32, device=dev)
    loss_out = None if reduction == "none" else torch.empty((), **f32)
    with torch.cuda.device(dev):
        ws_bytes = abi.flce_kl_forward_workspace_size(prob)
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev).cuda_stream
        abi.flce_kl_forward(prob, _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(target_probs),
                            _ptr(labels), _ptr(loss_rows), _ptr(lse_rows), _ptr(qsum_rows),
                            _ptr(loss_out), _ptr(n_counted), _ptr(err_word), _ptr(ws), ws_bytes,
                            stream)
    return {"loss": loss_rows if reduction == "none" else loss_out, "loss_rows": loss_rows,
            "lse_rows": lse_rows, "qsum_rows": qsum_rows, "n_counted": n_counted}


def flce_kl_backward_tensors(hidden, weight, target_probs, lse_rows, qsum_rows, n_counted,
                             grad_out, labels=None, bias=None, ignore_index=-100,
                             temperature=1.0, eps=1e-10, reduction="batchmean",
                             grad_weight_dtype=None, err_word=None, vocab_chunk=0,
                             skip_ignored=False):
    """Run flce_kl_backward; returns (grad_hidden, grad_weight, grad_bias)."""
    _check_kl_inputs(hidden, weight, target_probs, labels, bias)
    n, h = hidden.shape
    v = weight.shape[0]
    dev = hidden.device
    gw_dtype = hidden.dtype if grad_weight_dtype is None else grad_weight_dtype
    gw_code = abi.FLCE_F32 if gw_dtype == torch.float32 else _dtype_code(hidden)
    prob = abi.make_kl_problem(n, h, v, _dtype_code(hidden), bias is not None, ignore_index,
                               temperature, eps, reduction, grad_weight_dtype=gw_code,
                               vocab_chunk=vocab_chunk, skip_ignored=skip_ignored)
    grad_out = grad_out.to(device=dev, dtype=torch.float32).contiguous()
    grad_hidden = torch.empty_like(hidden)
    grad_weight = torch.empty(v, h, dtype=gw_dtype, device=dev)
    grad_bias = torch.empty_like(bias) if bias is not None else None
    with torch.cuda.device(dev):
        ws_bytes = abi.flce_kl_backward_workspace_size(prob)
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev).cuda_stream
        abi.flce_kl_backward(prob, _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(target_probs),
                             _ptr(labels), _ptr(lse_rows), _ptr(qsum_rows), _ptr(n_counted),
                             _ptr(grad_out), _ptr(grad_hidden), _ptr(grad_weight),
                             _ptr(grad_bias), _ptr(err_word), _ptr(ws), ws_bytes, stream)
    return grad_hidden, grad_weight, grad_bias


class _FusedLinearKLDiv(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, weight, bias, target_probs, labels, ignore_index, temperature, eps,
                reduction, vocab_chunk):
        out = flce_kl_forward_tensors(hidden, weight, target_probs, labels, bias, ignore_index,
                                      temperature, eps, reduction, skip_ignored=True)
        ctx.save_for_backward(hidden, weight, bias, target_probs, labels, out["lse_rows"],
                              out["qsum_rows"], out["n_counted"])
        ctx.opts = (ignore_index, temperature, eps, reduction, vocab_chunk)
        return out["loss"]

    @staticmethod
    def backward(ctx, grad_loss):
        hidden, weight, bias, target_probs, labels, lse_rows, qsum_rows, n_counted = \
            ctx.saved_tensors
        ignore_index, temperature, eps, reduction, vocab_chunk = ctx.opts
        gh, gw, gb = flce_kl_backward_tensors(hidden, weight, target_probs, lse_rows, qsum_rows,
                                              n_counted, grad_loss, labels, bias, ignore_index,
                                              temperature, eps, reduction, skip_ignored=True,
                                              vocab_chunk=vocab_chunk)
        need = ctx.needs_input_grad
        return (gh if need[0] else None, gw if need[1] else None,
                gb if (bias is not None and need[2]) else None,
                None, None, None, None, None, None, None)


def fused_linear_kl_div(hidden: torch.Tensor, weight: torch.Tensor,
                        target_probs: torch.Tensor, labels: Optional[torch.Tensor] = None,
                        bias: Optional[torch.Tensor] = None, ignore_index: int = -100,
                        temperature: float = 1.0, eps: float = 1e-10,
                        reduction: str = "batchmean", *, vocab_chunk: int = 0):
    """KL(target || softmax((hidden @ weight.T + bias) / temperature)) per row,
    reduced like torch.nn.KLDivLoss ('batchmean', 'mean', 'sum', 'none'),
    without materialising the (N, V) logits. hidden [..., H] may carry
    leading batch dimensions, matched by target_probs [..., V] and labels. Rows whose label equals
    ignore_index are left out (labels None: every row counts). The teacher
    probabilities get no gradient. ``vocab_chunk`` bounds the backward's
    dlogits buffer as in fused_linear_cross_entropy."""
    if reduction not in abi.KL_REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(abi.KL_REDUCTIONS)}")
    batch_shape = hidden.shape[:-1]
    if hidden.dim() > 2:  # leading batch dimensions: rows are flattened
        if target_probs.shape[:-1] != batch_shape or (
                labels is not None and labels.shape != batch_shape):
            raise ValueError("hidden [..., H], target_probs [..., V] and labels [...] must "
                             "share the leading shape")
        hidden = hidden.reshape(-1, hidden.shape[-1])
        target_probs = target_probs.reshape(-1, target_probs.shape[-1])
        labels = None if labels is None else labels.reshape(-1)
    hidden = hidden.contiguous()
    weight = weight.contiguous()
    target_probs = target_probs.detach().contiguous()
    labels = None if labels is None else labels.contiguous()
    bias = None if bias is None else bias.contiguous()
    loss = _FusedLinearKLDiv.apply(hidden, weight, bias, target_probs, labels,
                                   int(ignore_index), float(temperature), float(eps), reduction,
                                   int(vocab_chunk))
    return loss.reshape(batch_shape) if reduction == "none" else loss
