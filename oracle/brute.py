"""Pure-Python brute force for tiny fused linear cross-entropy problems.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see ``oracle/__init__.py``).

It materialises every logit as a Python float (IEEE fp64), normalises the
softmax explicitly (no max shift, no log-sum-exp identity) and takes the
forward quantities from their textbook forms:

  * loss_i = -log p_{i,t_i} with p = exp(z) / sum(exp(z));
  * entropy_i = -sum_j p_ij log p_ij;
  * argmax_i = the lowest j with the largest z_ij.

It shares no code with :mod:`oracle.flce_oracle`: it exists to pin that
module (which uses the max-shifted log-sum-exp, ``lse - sum p z`` for the
entropy, and a library matmul). Gradients are pinned separately by central
finite differences of :func:`loss` below. Inputs must be small (a few
thousand logits) and moderate in value so that exp() does not overflow.

Follows "fused-linear-ce" (trl-lib model card), §Full signature, §Metrics for
free and §Algorithm, with the same readings as the streaming oracle.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence


def _logit(h: Sequence[float], w: Sequence[float], b: Optional[float],
           logit_scale: float, softcap: Optional[float]) -> float:
    acc = 0.0
    for x, y in zip(h, w):
        acc += float(x) * float(y)
    if b is not None:
        acc += float(b)
    u = logit_scale * acc
    if softcap is not None and softcap > 0:
        return softcap * math.tanh(u / softcap)
    return u


def logits(hidden, weight, bias, logit_scale=1.0, softcap=None) -> List[List[float]]:
    """All N x V final logits as nested lists of Python floats."""
    out = []
    for h in hidden:
        row = []
        for j, w in enumerate(weight):
            row.append(_logit(h, w, None if bias is None else bias[j],
                              logit_scale, softcap))
        out.append(row)
    return out


def per_row(hidden, weight, targets, bias=None, ignore_index=-100,
            logit_scale=1.0, softcap=None, label_smoothing=0.0,
            z_loss=0.0) -> List[dict]:
    """Per-row loss, entropy, argmax and validity by explicit softmax.

    With label smoothing eps the loss is the cross-entropy against the target
    distribution q = (1-eps)*onehot + eps/V, -sum_j q_j log p_j; with z_loss
    lam, lam * (log sum_j e^{z_j})^2 is added (the options named in the
    CuTe-DSL FLCE pull request's feature list)."""
    z_all = logits(hidden, weight, bias, logit_scale, softcap)
    v = len(weight)
    rows = []
    for z, t in zip(z_all, targets):
        t = int(t)
        e = [math.exp(x) for x in z]
        tot = sum(e)
        p = [x / tot for x in e]
        ent = 0.0
        for q in p:
            if q > 0.0:
                ent -= q * math.log(q)
        best = 0
        for j in range(1, v):
            if z[j] > z[best]:
                best = j
        valid = t != ignore_index
        if not valid:
            loss = 0.0
        elif 0 <= t < v:
            loss = 0.0
            for j in range(v):
                q = (1.0 - label_smoothing) * (1.0 if j == t else 0.0) + label_smoothing / v
                if q != 0.0:
                    loss -= q * math.log(p[j])
            if z_loss != 0.0:
                loss += z_loss * math.log(tot) ** 2
        else:
            loss = float("nan")
        rows.append({"loss": loss, "entropy": ent, "argmax": best,
                     "valid": valid, "correct": valid and best == t,
                     "p": p})
    return rows


def loss(hidden, weight, targets, bias=None, ignore_index=-100,
         logit_scale=1.0, softcap=None, reduction="mean", row_grads=None,
         label_smoothing=0.0, z_loss=0.0):
    """Reduced loss. For reduction 'none' the per-row losses are combined with
    ``row_grads`` (a scalar objective sum_i row_grads[i] * loss_i) so that
    finite differences can probe the per-row upstream-gradient path."""
    rows = per_row(hidden, weight, targets, bias, ignore_index, logit_scale,
                   softcap, label_smoothing, z_loss)
    n_valid = sum(1 for r in rows if r["valid"])
    tot = sum(r["loss"] for r in rows)
    if reduction == "sum":
        return tot
    if reduction == "mean":
        return tot / n_valid if n_valid else float("nan")
    if reduction == "none":
        if row_grads is None:
            return [r["loss"] for r in rows]
        return sum(g * r["loss"] for g, r in zip(row_grads, rows))
    raise ValueError(reduction)


def metrics(hidden, weight, targets, bias=None, ignore_index=-100,
            logit_scale=1.0, softcap=None):
    """(mean_token_accuracy, mean entropy) over non-ignored rows."""
    rows = per_row(hidden, weight, targets, bias, ignore_index, logit_scale,
                   softcap)
    val = [r for r in rows if r["valid"]]
    if not val:
        return float("nan"), float("nan")
    acc = sum(1 for r in val if r["correct"]) / len(val)
    ent = sum(r["entropy"] for r in val) / len(val)
    return acc, ent


def kl_per_row(hidden, weight, target_probs, bias=None, labels=None, ignore_index=-100,
               temperature=1.0, eps=1e-10):
    """Per-row KL(Q || P) by explicit softmax of the logits / T:
    sum_j q_j (log max(q_j, eps) - log p_j), 0 for ignored rows (the fused
    linear KL divergence of Liger-Kernel pull request #1423)."""
    z_all = logits(hidden, weight, bias, 1.0 / temperature, None)
    out = []
    for i, (z, q) in enumerate(zip(z_all, target_probs)):
        if labels is not None and int(labels[i]) == ignore_index:
            out.append(0.0)
            continue
        e = [math.exp(x) for x in z]
        tot = sum(e)
        acc = 0.0
        for qj, ej in zip(q, e):
            qj = float(qj)
            acc += qj * (math.log(max(qj, eps)) - math.log(ej / tot))
        out.append(acc)
    return out


def kl_loss(hidden, weight, target_probs, bias=None, labels=None, ignore_index=-100,
            temperature=1.0, eps=1e-10, reduction="batchmean", row_grads=None):
    rows = kl_per_row(hidden, weight, target_probs, bias, labels, ignore_index, temperature,
                      eps)
    n_counted = len(rows) if labels is None else sum(1 for t in labels if int(t) != ignore_index)
    tot = sum(rows)
    if reduction == "sum":
        return tot
    if reduction == "batchmean":
        return tot / n_counted
    if reduction == "mean":
        return tot / (n_counted * len(weight))
    if reduction == "none":
        return sum(g * r for g, r in zip(row_grads, rows))
    raise ValueError(reduction)
