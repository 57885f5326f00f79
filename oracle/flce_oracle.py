"""Plain fp64 CPU oracle for fused linear cross-entropy.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import or run anything in ``oracle/``. The library's own path
never calls it, and it shares no code with the CUDA kernels.

What it computes follows the "fused-linear-ce" model card (trl-lib):
  * §Full signature: ``fused_linear_cross_entropy(hidden (N,H), weight (V,H),
    targets (N,), bias=None, ignore_index=-100, logit_scale=1.0, softcap=None,
    reduction="mean"|"sum"|"none", return_metrics=False)``; hidden, weight
    and bias all receive gradients.
  * §Metrics for free: ``mean_token_accuracy`` is the fraction of
    non-ignored positions whose argmax logit is the target; ``entropy`` is the
    mean softmax entropy in nats.
  * §Algorithm: logits ``hidden @ weight.T`` with bias, logit_scale and
    softcap applied in that order; cross-entropy through the log-sum-exp; the
    backward forms ``p - onehot`` and takes ``grad_hidden = (p - onehot) @
    weight`` and ``grad_weight = (p - onehot).T @ hidden``.

This is the plain definition: every logit is formed in fp64 from the exactly
widened inputs, each row's softmax statistics are taken over the whole row,
and the gradients are the chain rule of that definition. Rows are processed in
blocks only to bound host memory; rows are independent, so the blocking does
not change what is computed. A library matmul serves as the dot-product step.

Readings where the card is silent (each is listed with its reason in the
design notes):
  * softcap ``c``: ``z = c * tanh(u / c)`` with ``u = logit_scale * (h.w + b)``;
    ``softcap`` None or <= 0 means off.
  * The gradient carries the chain factor ``logit_scale * (1 - tanh(u/c)^2)``
    (the exact derivative of the definition); logit_scale and softcap get no
    gradient.
  * ``mean`` divides by n_valid, the number of rows whose target is not
    ignore_index; n_valid = 0 gives NaN loss and metrics and zero gradients.
  * ``none`` returns per-row losses (0 on ignored rows); its backward takes a
    per-row upstream gradient.
  * Metrics are means over non-ignored rows for every reduction; argmax ties
    go to the lowest vocabulary index.
  * A target outside [0, V) that is not ignore_index counts as non-ignored,
    gets a NaN loss, is never "correct", and contributes no gradient.

Two options from the feature list of the CuTe-DSL FLCE pull request
(Liger-Kernel #1287, §Summary, which lists z-loss, softcap and label smoothing
among its options),
which names them without defining them; the readings taken:
  * label_smoothing eps: the target distribution is (1-eps)*onehot + eps/V,
    so loss_i = (1-eps)*(lse_i - z_{i,t_i}) + eps*(lse_i - mean_j z_ij);
  * z_loss lam: lam * lse_i^2 is added to each non-ignored row's loss;
and the gradient with respect to z_ij is
    g_i * [p_ij*(1 + 2*lam*lse_i) - (1-eps)*[j == t_i] - eps/V].
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

__all__ = [
    "final_logits",
    "forward",
    "backward",
    "row_weights",
    "valid_mask",
]

_F64 = torch.float64


def _softcap_on(softcap: Optional[float]) -> bool:
    return softcap is not None and softcap > 0


def final_logits(h_rows: torch.Tensor, weight: torch.Tensor,
                 bias: Optional[torch.Tensor], logit_scale: float,
                 softcap: Optional[float]):
    """Final logits z and the pre-softcap values u for a block of rows.

    u = logit_scale * (h @ W^T + b);  z = softcap * tanh(u / softcap) when a
    softcap is given, else z = u ("fused-linear-ce", §Algorithm: bias /
    logit_scale / softcap applied in that order). All in fp64.
    """
    lin = h_rows.to(_F64) @ weight.to(_F64).T
    if bias is not None:
        lin = lin + bias.to(_F64)
    u = logit_scale * lin
    if _softcap_on(softcap):
        z = softcap * torch.tanh(u / softcap)
    else:
        z = u
    return z, u


def valid_mask(targets: torch.Tensor, ignore_index: int) -> torch.Tensor:
    """Rows that are not ignored (§Metrics for free: 'over non-ignored
    positions')."""
    return targets != ignore_index


def _in_range(targets: torch.Tensor, v: int) -> torch.Tensor:
    return (targets >= 0) & (targets < v)


def _row_block(v: int, budget_bytes: int = 256 << 20) -> int:
    return max(1, min(4096, budget_bytes // (8 * max(v, 1) * 3)))


def forward(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
            bias: Optional[torch.Tensor] = None, ignore_index: int = -100,
            logit_scale: float = 1.0, softcap: Optional[float] = None,
            reduction: str = "mean",
            rows: Optional[Sequence[int]] = None,
            label_smoothing: float = 0.0, z_loss: float = 0.0) -> dict:
    """Forward of the loss in fp64.

    Returns per-row ``loss``, ``lse``, ``argmax``, ``entropy``,
    ``target_logit``, ``max_logit``, ``top2_gap`` (gap between the two largest
    logits) and ``correct`` for the selected rows (all rows when ``rows`` is None), and,
    when all rows are computed, the reduced ``loss_out``,
    ``mean_token_accuracy`` and ``entropy_mean``. ``n_valid`` and
    ``target_error`` (a target out of range that is not ignore_index) are
    always over all rows.
    """
    n, _ = hidden.shape
    v = weight.shape[0]
    targets = targets.to(torch.int64)
    valid_all = valid_mask(targets, ignore_index)
    n_valid = int(valid_all.sum())
    target_error = bool((valid_all & ~_in_range(targets, v)).any())

    # widen once; every logit below is formed from these exact fp64 copies
    weight = weight.to(_F64)
    bias = None if bias is None else bias.to(_F64)
    idx = torch.arange(n) if rows is None else torch.as_tensor(list(rows), dtype=torch.int64)
    k = idx.numel()
    out = {name: torch.empty(k, dtype=_F64) for name in
           ("loss", "lse", "entropy", "target_logit", "max_logit", "top2_gap")}
    out["argmax"] = torch.empty(k, dtype=torch.int64)
    blk = _row_block(v)
    for s in range(0, k, blk):
        ri = idx[s:s + blk]
        z, _ = final_logits(hidden[ri], weight, bias, logit_scale, softcap)
        # row maximum and its lowest index
        m = z.max(dim=1).values
        am = torch.argmax(z, dim=1)
        lse = m + torch.log(torch.exp(z - m[:, None]).sum(dim=1))
        p = torch.exp(z - lse[:, None])
        # entropy H = -sum p log p = lse - sum p z
        ent = lse - (p * z).sum(dim=1)
        t = targets[ri]
        ok = _in_range(t, v)
        zt = torch.full((ri.numel(),), float("nan"), dtype=_F64)
        zt[ok] = z[torch.nonzero(ok).flatten(), t[ok]]
        loss = lse - zt
        if label_smoothing != 0.0:
            # cross-entropy against (1-eps)*onehot + eps/V
            loss = (1.0 - label_smoothing) * loss + label_smoothing * (lse - z.mean(dim=1))
        if z_loss != 0.0:
            loss = loss + z_loss * lse * lse
        vm = valid_mask(t, ignore_index)
        loss = torch.where(vm, loss, torch.zeros_like(loss))
        if v >= 2:
            top2 = torch.topk(z, 2, dim=1).values
            gap = top2[:, 0] - top2[:, 1]
        else:
            gap = torch.full((ri.numel(),), float("inf"), dtype=_F64)
        out["loss"][s:s + blk] = loss
        out["lse"][s:s + blk] = lse
        out["entropy"][s:s + blk] = ent
        out["argmax"][s:s + blk] = am
        out["target_logit"][s:s + blk] = zt
        out["max_logit"][s:s + blk] = m
        out["top2_gap"][s:s + blk] = gap
    t_sel = targets[idx]
    vm_sel = valid_mask(t_sel, ignore_index)
    out["valid"] = vm_sel
    out["correct"] = vm_sel & (out["argmax"] == t_sel)
    out["rows"] = idx
    out["n_valid"] = n_valid
    out["target_error"] = target_error
    if rows is None:
        nan = float("nan")
        tot = float(out["loss"].sum())
        if reduction == "none":
            out["loss_out"] = out["loss"].clone()
        elif reduction == "sum":
            out["loss_out"] = tot
        elif reduction == "mean":
            out["loss_out"] = tot / n_valid if n_valid > 0 else nan
        else:
            raise ValueError(f"unknown reduction {reduction!r}")
        if n_valid > 0:
            out["mean_token_accuracy"] = float(out["correct"].sum()) / n_valid
            out["entropy_mean"] = float(out["entropy"][vm_sel].sum()) / n_valid
        else:
            out["mean_token_accuracy"] = nan
            out["entropy_mean"] = nan
    return out


def row_weights(targets: torch.Tensor, v: int, ignore_index: int,
                reduction: str, grad_out) -> torch.Tensor:
    """Upstream gradient g_i of each row's loss term: grad_out / n_valid for
    'mean', grad_out for 'sum', grad_out[i] for 'none'; 0 on ignored rows and
    on rows whose target is out of range."""
    targets = targets.to(torch.int64)
    vm = valid_mask(targets, ignore_index)
    n_valid = int(vm.sum())
    live = vm & _in_range(targets, v)
    if reduction == "none":
        g = torch.as_tensor(grad_out, dtype=_F64).reshape(-1).clone()
    elif reduction == "sum":
        g = torch.full((targets.numel(),), float(grad_out), dtype=_F64)
    elif reduction == "mean":
        scale = float(grad_out) / n_valid if n_valid > 0 else 0.0
        g = torch.full((targets.numel(),), scale, dtype=_F64)
    else:
        raise ValueError(f"unknown reduction {reduction!r}")
    return torch.where(live, g, torch.zeros_like(g))


def _dlogits(z: torch.Tensor, u: torch.Tensor, lse: torch.Tensor,
             pos: torch.Tensor, g: torch.Tensor, logit_scale: float,
             softcap: Optional[float], label_smoothing: float = 0.0,
             z_loss: float = 0.0, v_total: int = 0) -> torch.Tensor:
    """d loss / d lin for a block:
    g_i * (p_ij*(1 + 2*z_loss*lse_i) - (1-eps)*[j == t_i] - eps/V) * dz/dlin
    (eps = label_smoothing; with both options off, g_i * (p_ij - [j == t_i])).

    ``pos[i]`` is the column of row i's target within ``z`` (or -1 when the
    target is not among these columns). dz/dlin = logit_scale * (1 -
    tanh(u/c)^2) with a softcap, else logit_scale.
    """
    d = torch.exp(z - lse[:, None])
    if z_loss != 0.0:
        d *= (1.0 + 2.0 * z_loss * lse)[:, None]
    hit = pos >= 0
    d[torch.nonzero(hit).flatten(), pos[hit]] -= 1.0 - label_smoothing
    if label_smoothing != 0.0:
        d -= label_smoothing / v_total
    d *= g[:, None]
    d *= logit_scale
    if _softcap_on(softcap):
        d *= 1.0 - torch.tanh(u / softcap) ** 2
    return d


def _abs_terms(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    """|a| @ |b|: entry (i, k) is the sum of the absolute values of the terms
    a_ij b_jk that make up (a @ b)_ik."""
    return a.abs() @ b.abs()


def backward(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
             bias: Optional[torch.Tensor] = None, ignore_index: int = -100,
             logit_scale: float = 1.0, softcap: Optional[float] = None,
             reduction: str = "mean", grad_out=1.0,
             lse: Optional[torch.Tensor] = None,
             rows: Optional[Sequence[int]] = None,
             vocab_rows: Optional[Sequence[int]] = None,
             want_hidden: bool = True, want_weight: bool = True,
             label_smoothing: float = 0.0, z_loss: float = 0.0,
             magnitudes: bool = False) -> dict:
    """Gradients of the loss in fp64 (§Algorithm: grad_hidden = (p - onehot)
    @ weight, grad_weight = (p - onehot).T @ hidden; bias gets the column
    sums), with the chain factor of logit_scale and softcap.

    ``rows`` restricts grad_hidden to those rows; ``vocab_rows`` restricts
    grad_weight and grad_bias to those vocabulary rows. ``lse`` (fp64 [N]) may
    be passed from :func:`forward` to avoid recomputing it; grad_weight needs
    the lse of every row.

    ``magnitudes`` also returns, for every gradient entry, the sum of the
    absolute values of the terms it adds up (``*_mag``):
    ``sum_j |D_ij| |W_jk|`` for grad_hidden, ``sum_i |D_ij| |h_ik|`` for
    grad_weight and ``sum_i |D_ij|`` for grad_bias, with D = d loss / d lin as
    above. Perturbing every D_ij by at most a fraction u of itself moves the
    entry by at most u times this sum, so it is the scale against which an
    implementation that rounds D (or accumulates the terms in finite
    precision) is judged. Test infrastructure; it does not enter the gradients.
    """
    n, _ = hidden.shape
    v = weight.shape[0]
    targets = targets.to(torch.int64)
    g_all = row_weights(targets, v, ignore_index, reduction, grad_out)
    weight = weight.to(_F64)
    bias = None if bias is None else bias.to(_F64)
    out = {}
    if want_hidden:
        idx = torch.arange(n) if rows is None else torch.as_tensor(list(rows), dtype=torch.int64)
        w64 = weight
        gh = torch.empty(idx.numel(), hidden.shape[1], dtype=_F64)
        gh_mag = torch.empty_like(gh) if magnitudes else None
        blk = _row_block(v)
        for s in range(0, idx.numel(), blk):
            ri = idx[s:s + blk]
            z, u = final_logits(hidden[ri], weight, bias, logit_scale, softcap)
            if lse is None:
                m = z.max(dim=1).values
                lse_b = m + torch.log(torch.exp(z - m[:, None]).sum(dim=1))
            else:
                lse_b = lse[ri].to(_F64)
            t = targets[ri]
            pos = torch.where(_in_range(t, v), t, torch.full_like(t, -1))
            d = _dlogits(z, u, lse_b, pos, g_all[ri], logit_scale, softcap,
                         label_smoothing, z_loss, v)
            gh[s:s + blk] = d @ w64
            if magnitudes:
                gh_mag[s:s + blk] = _abs_terms(d, w64)
        out["grad_hidden"] = gh
        out["rows"] = idx
        if magnitudes:
            out["grad_hidden_mag"] = gh_mag
    if want_weight:
        if lse is None:
            lse = forward(hidden, weight, targets, bias, ignore_index,
                          logit_scale, softcap, reduction)["lse"]  # lse needs no options
        jdx = torch.arange(v) if vocab_rows is None else torch.as_tensor(list(vocab_rows), dtype=torch.int64)
        # column of each vocabulary id among the selected rows, -1 if absent
        col_of = torch.full((v,), -1, dtype=torch.int64)
        col_of[jdx] = torch.arange(jdx.numel())
        if vocab_rows is None:
            w_sel, b_sel = weight, bias
        else:
            w_sel = weight[jdx]
            b_sel = None if bias is None else bias[jdx]
        gw = torch.zeros(jdx.numel(), hidden.shape[1], dtype=_F64)
        gb = torch.zeros(jdx.numel(), dtype=_F64)
        gw_mag = torch.zeros_like(gw) if magnitudes else None
        gb_mag = torch.zeros_like(gb) if magnitudes else None
        blk = _row_block(jdx.numel())
        for s in range(0, n, blk):
            ri = torch.arange(s, min(n, s + blk))
            z, u = final_logits(hidden[ri], w_sel, b_sel, logit_scale, softcap)
            t = targets[ri]
            pos = torch.full_like(t, -1)
            ok = _in_range(t, v)
            pos[ok] = col_of[t[ok]]
            d = _dlogits(z, u, lse[ri].to(_F64), pos, g_all[ri], logit_scale,
                         softcap, label_smoothing, z_loss, v)
            gw += d.T @ hidden[ri].to(_F64)
            gb += d.sum(dim=0)
            if magnitudes:
                gw_mag += _abs_terms(d.T, hidden[ri].to(_F64))
                gb_mag += d.abs().sum(dim=0)
        out["grad_weight"] = gw
        out["grad_bias"] = gb if bias is not None else None
        out["vocab_rows"] = jdx
        if magnitudes:
            out["grad_weight_mag"] = gw_mag
            out["grad_bias_mag"] = gb_mag if bias is not None else None
    return out
