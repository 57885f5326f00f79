"""Plain fp64 CPU oracle for the fused linear KL divergence.

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import or run it. It shares no code with the CUDA path.

What it computes follows the FusedLinearKLDivLoss pull request (Liger-Kernel
#1423), §Summary and §Details: the vocabulary projection of the student's
hidden states, then KL(Q || P) against an explicit target distribution Q
(teacher probabilities), with softmax temperature T, an eps clamp so that
0 * log 0 contributes 0, reductions "batchmean" / "mean" / "sum" with the
semantics of torch.nn.KLDivLoss, and ignored rows. Per row i:

    z_ij   = (h_i . w_j + b_j) / T
    log p_ij = z_ij - lse_i,     lse_i = log sum_j e^{z_ij}
    loss_i = sum_j q_ij * (log max(q_ij, eps) - log p_ij)

(the pull request's in-kernel commit evaluates it in the equal factored form
sum_j q_ij (log max(q_ij, eps) - z_ij) + lse_i * sum_j q_ij; this oracle
takes the definition above directly). Gradient with respect to z_ij:
p_ij * sum_k q_ik - q_ij; with respect to the linear logits it carries the
1/T factor.

Readings where the pages are silent:
  * ignored rows: a row whose label equals ignore_index contributes no loss
    and no gradient (the pull request handles ignore_index through its
    shifted labels);
    without labels every row counts;
  * "batchmean" divides the summed loss by the number of counted rows,
    "mean" by that number times V (torch.nn.KLDivLoss divides by the batch
    size and by the element count, with every row counted);
  * reduction "none" (refused by the pull request only because its gradient
    is formed during the forward) returns per-row losses and takes a per-row
    upstream gradient;
  * no T^2 factor is applied to the loss.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

__all__ = ["forward", "backward", "row_weights"]

_F64 = torch.float64


def _counted(labels: Optional[torch.Tensor], n: int, ignore_index: int) -> torch.Tensor:
    if labels is None:
        return torch.ones(n, dtype=torch.bool)
    return labels.to(torch.int64) != ignore_index


def _row_block(v: int, budget_bytes: int = 256 << 20) -> int:
    return max(1, min(4096, budget_bytes // (8 * max(v, 1) * 4)))


def _logits(h_rows, weight64, bias64, temperature):
    lin = h_rows.to(_F64) @ weight64.T
    if bias64 is not None:
        lin = lin + bias64
    return lin / temperature


def forward(hidden: torch.Tensor, weight: torch.Tensor, target_probs: torch.Tensor,
            bias: Optional[torch.Tensor] = None, labels: Optional[torch.Tensor] = None,
            ignore_index: int = -100, temperature: float = 1.0, eps: float = 1e-10,
            reduction: str = "batchmean",
            rows: Optional[Sequence[int]] = None) -> dict:
    """Per-row ``loss``, ``lse`` (of z = logits / T) and ``qsum`` (sum_j q_ij)
    for the selected rows (all when ``rows`` is None), and, for all rows, the
    reduced ``loss_out``. ``n_counted`` is the number of counted rows."""
    n = hidden.shape[0]
    v = weight.shape[0]
    counted = _counted(labels, n, ignore_index)
    n_counted = int(counted.sum())
    w64 = weight.to(_F64)
    b64 = None if bias is None else bias.to(_F64)
    idx = torch.arange(n) if rows is None else torch.as_tensor(list(rows), dtype=torch.int64)
    out = {k: torch.empty(idx.numel(), dtype=_F64) for k in ("loss", "lse", "qsum")}
    blk = _row_block(v)
    for s in range(0, idx.numel(), blk):
        ri = idx[s:s + blk]
        z = _logits(hidden[ri], w64, b64, temperature)
        m = z.max(dim=1).values
        lse = m + torch.log(torch.exp(z - m[:, None]).sum(dim=1))
        logp = z - lse[:, None]
        q = target_probs[ri].to(_F64)
        loss = (q * (torch.log(torch.clamp(q, min=eps)) - logp)).sum(dim=1)
        loss = torch.where(counted[ri], loss, torch.zeros_like(loss))
        out["loss"][s:s + blk] = loss
        out["lse"][s:s + blk] = lse
        out["qsum"][s:s + blk] = q.sum(dim=1)
    out["rows"] = idx
    out["counted"] = counted[idx]
    out["n_counted"] = n_counted
    if rows is None:
        tot = float(out["loss"].sum())
        nan = float("nan")
        if reduction == "none":
            out["loss_out"] = out["loss"].clone()
        elif reduction == "sum":
            out["loss_out"] = tot
        elif reduction == "batchmean":
            out["loss_out"] = tot / n_counted if n_counted else nan
        elif reduction == "mean":
            out["loss_out"] = tot / (n_counted * v) if n_counted else nan
        else:
            raise ValueError(f"unknown reduction {reduction!r}")
    return out


def row_weights(labels, n: int, v: int, ignore_index: int, reduction: str, grad_out) -> torch.Tensor:
    """Upstream gradient of each row's loss term; 0 on ignored rows."""
    counted = _counted(labels, n, ignore_index)
    nc = int(counted.sum())
    if reduction == "none":
        g = torch.as_tensor(grad_out, dtype=_F64).reshape(-1).clone()
    elif reduction == "sum":
        g = torch.full((n,), float(grad_out), dtype=_F64)
    elif reduction == "batchmean":
        g = torch.full((n,), float(grad_out) / nc if nc else 0.0, dtype=_F64)
    elif reduction == "mean":
        g = torch.full((n,), float(grad_out) / (nc * v) if nc else 0.0, dtype=_F64)
    else:
        raise ValueError(f"unknown reduction {reduction!r}")
    return torch.where(counted, g, torch.zeros_like(g))


def _abs_terms(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    """|a| @ |b|: the sums of the absolute values of the terms of a @ b."""
    return a.abs() @ b.abs()


def backward(hidden: torch.Tensor, weight: torch.Tensor, target_probs: torch.Tensor,
             bias: Optional[torch.Tensor] = None, labels: Optional[torch.Tensor] = None,
             ignore_index: int = -100, temperature: float = 1.0, eps: float = 1e-10,
             reduction: str = "batchmean", grad_out=1.0,
             rows: Optional[Sequence[int]] = None,
             vocab_rows: Optional[Sequence[int]] = None,
             magnitudes: bool = False) -> dict:
    """grad_hidden (selected rows), grad_weight and grad_bias (selected
    vocabulary rows) in fp64: with D_ij = g_i (p_ij sum_k q_ik - q_ij) / T,
    grad_hidden = D @ W, grad_weight = D^T @ H, grad_bias = sum_i D_ij.

    ``magnitudes`` also returns the sums of the absolute values of each
    entry's terms (``*_mag``: sum_j |D_ij||W_jk|, sum_i |D_ij||h_ik|,
    sum_i |D_ij|), the scale against which rounding D is judged (as in the
    cross-entropy oracle). Test infrastructure; the gradients are unchanged."""
    n = hidden.shape[0]
    v = weight.shape[0]
    g_all = row_weights(labels, n, v, ignore_index, reduction, grad_out)
    w64 = weight.to(_F64)
    b64 = None if bias is None else bias.to(_F64)
    idx = torch.arange(n) if rows is None else torch.as_tensor(list(rows), dtype=torch.int64)
    jdx = torch.arange(v) if vocab_rows is None else torch.as_tensor(list(vocab_rows), dtype=torch.int64)
    gh = torch.empty(idx.numel(), hidden.shape[1], dtype=_F64)
    gw = torch.zeros(jdx.numel(), hidden.shape[1], dtype=_F64)
    gb = torch.zeros(jdx.numel(), dtype=_F64)
    gh_mag = torch.empty_like(gh) if magnitudes else None
    gw_mag = torch.zeros_like(gw) if magnitudes else None
    gb_mag = torch.zeros_like(gb) if magnitudes else None
    blk = _row_block(v)
    pos_of = torch.full((n,), -1, dtype=torch.int64)  # position of each row among `rows`
    pos_of[idx] = torch.arange(idx.numel())
    for s in range(0, n, blk):
        ri = torch.arange(s, min(n, s + blk))
        z = _logits(hidden[ri], w64, b64, temperature)
        m = z.max(dim=1).values
        lse = m + torch.log(torch.exp(z - m[:, None]).sum(dim=1))
        p = torch.exp(z - lse[:, None])
        q = target_probs[ri].to(_F64)
        d = (p * q.sum(dim=1)[:, None] - q) * (g_all[ri] / temperature)[:, None]
        gw += d[:, jdx].T @ hidden[ri].to(_F64)
        gb += d[:, jdx].sum(dim=0)
        pos = pos_of[ri]
        take = pos >= 0
        gh[pos[take]] = d[take] @ w64
        if magnitudes:
            gw_mag += _abs_terms(d[:, jdx].T, hidden[ri].to(_F64))
            gb_mag += d[:, jdx].abs().sum(dim=0)
            gh_mag[pos[take]] = _abs_terms(d[take], w64)
    out = {"grad_hidden": gh, "grad_weight": gw,
           "grad_bias": gb if bias is not None else None, "rows": idx, "vocab_rows": jdx}
    if magnitudes:
        out["grad_hidden_mag"] = gh_mag
        out["grad_weight_mag"] = gw_mag
        out["grad_bias_mag"] = gb_mag if bias is not None else None
    return out
