"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 oracle on the same seeded inputs.

Every bar is stated in the units of the output it checks, for every
reduction (no rescaling of 'sum' or 'none' results).

Per-row loss, lse and entropy (and the KL divergence's per-row loss):
    |got - ref| <= rel * |ref| + floor_i
with rel 1e-5 for fp32 inputs and 2e-3 for 16-bit inputs, and
    floor_i = (ceil(H/16) + 8) * 2^-24 * ops_i,
    ops_i   = |lse_i| + |max_j z_ij| + |z_{i,t_i}|   (cross-entropy)
              |lse_i| * Q_i + |loss_i - lse_i * Q_i|  (KL, Q_i = sum_j q_ij)
The floor is the fp32 evaluation of those operands: a logit is an fp32 sum
of H products, accumulated in ceil(H/16) rounded steps on the tensor cores
(one per 16-product MMA step; their rounding mode is not assumed unbiased,
so the errors may add up linearly), plus a few rounded operations for the
maximum, the exponentials, their sum and the logarithm. The fp32 path rounds
after each of its H fused multiply-adds to nearest even, whose errors grow
like sqrt(H) <= ceil(H/16) + 8 for every H. Without a floor a 'relative' bar
would ask a row whose loss is 1e-4 (a confident row) for a result more exact
than the fp32 rounding of its own lse. The reduced loss gets the matching
bar: rel * |ref| plus the mean (or the sum) of the rows' floors plus the
fp32 rounding of its own tree sum, (ceil(log2 N) + 1) * 2^-24 * sum |loss_i|.

Gradients, elementwise:
    |got - ref| <= atol + rtol * |ref| + floor + kappa * M
with (atol, rtol) = (5e-5, 5e-2) for bf16 and (1e-5, 1e-4) for fp32, and M
the oracle's sum of the absolute values of the entry's terms
(sum_j |D_ij||W_jk| for grad_hidden, sum_i |D_ij||h_ik| for grad_weight,
sum_i |D_ij| for grad_bias; D = d loss / d lin). kappa bounds the relative
perturbation of each term:
  * u_D, the rounding of D to the GEMM operand type: 2^-8 for bf16 and
    2^-11 for fp16 (round to nearest even with 8 and 11 significant bits), 0
    for fp32 (D stays fp32) and 0 for grad_bias (summed from the fp32 D);
  * the fp32 accumulation of the K terms: tensor cores round once per
    16-product MMA step, up to one unit (2^-23) each, over ceil(K/16) steps
    plus one per vocabulary chunk (grad_hidden adds chunks in fp32); the fp32
    path rounds each of its K steps to nearest (2^-24); grad_bias adds
    ceil(N/128) partial sums of shuffle trees of 128 rows.
    K = V for grad_hidden, K = N for grad_weight.
Where terms cancel (vocabulary rows hit by several targets, peaked rows, a
sharp temperature) the exact entry is small while rounding each term still
moves it by up to u_D times that term, so an entry's error is bounded by
kappa * M, not by a multiple of the entry itself. fp16 outputs widen both
bars by 2^-25 (``g_floor``): a gradient below fp16's smallest normal value
(2^-14) is stored as a subnormal, spaced 2^-24 apart, whatever the kernel
computed.

Gradients, normwise: ||got - ref|| / ||ref|| <= 1e-2 (16-bit) / 1e-4
(fp32). At mean scale gradients are ~1e-6 and the elementwise atol alone
would pass a wrong factor; the normwise bar catches it.

Argmax-based correctness: bit-exact on rows whose oracle top-2 logit gap
exceeds 1e-2.
"""
from __future__ import annotations

import math

import torch

import oracle
from linear_cross_entropy_vocab_gb300 import api

TOL = {
    "f32": dict(loss_rel=1e-5, g_atol=1e-5, g_rtol=1e-4, g_norm=1e-4, ent_rel=1e-4, u_d=0.0,
                acc_unit=2.0 ** -24, acc_k=1),
    "bf16": dict(loss_rel=2e-3, g_atol=5e-5, g_rtol=5e-2, g_norm=1e-2, ent_rel=1e-3,
                 u_d=2.0 ** -8, acc_unit=2.0 ** -23, acc_k=16),
}
# fp16 inputs: the pages state no fp16 bar. fp16 rounds more finely than bf16
# (2^-11 against 2^-8 relative) in every place the bf16 path rounds (D and the
# outputs), so the bf16 bars bound the fp16 path, except where fp16's narrow
# exponent range bites: gradients stored in fp16 below its smallest normal
# value (2^-14) are subnormal, spaced 2^-24 apart, so rounding an output there
# errs by up to 2^-25 absolute whatever the kernel does (a 'mean' KL divergence
# divides by N*V and lands there). ``g_floor`` adds that half-spacing to the
# elementwise and normwise bars.
TOL["f16"] = dict(TOL["bf16"], g_floor=2.0 ** -25, u_d=2.0 ** -11)

U24 = 2.0 ** -24


def row_floor(h: int, ops):
    """Absolute floor of the per-row bars: (ceil(H/16) + 8) fp32 units of the
    operands' magnitude ``ops`` (see the module docstring)."""
    return (math.ceil(h / 16) + 8) * U24 * ops


def ce_row_ops(ref):
    """|lse| + |max logit| + |target logit| per row of an oracle forward."""
    return (ref["lse"].abs() + ref["max_logit"].abs()
            + ref["target_logit"].nan_to_num(0.0).abs())


def kl_row_ops(ref):
    """|lse| Q + |loss - lse Q| per row of a KL oracle forward (Q = sum q)."""
    lq = ref["lse"] * ref["qsum"]
    return lq.abs() + (ref["loss"] - lq).abs()


def kappa(tol, k: int, chunks: int = 0) -> float:
    """Relative perturbation bound of each term of a gradient entry that sums
    k terms: the rounding of D to the operand type plus the fp32 accumulation
    (see the module docstring); ``chunks`` more fp32 additions."""
    steps = math.ceil(k / tol["acc_k"]) + chunks + 8
    return tol["u_d"] + steps * tol["acc_unit"]


def bias_kappa(n: int) -> float:
    """grad_bias: fp32 column sums of the unrounded fp32 D, shuffle trees over
    128-row tiles (8 steps) then ceil(N/128) partial sums in a fixed order."""
    return (math.ceil(n / 128) + 16) * U24


def grad_kappas(w, n_rows: int = None) -> dict:
    """kappa of each gradient of a cross-entropy or KL problem of the shape of
    workload ``w`` (``n_rows`` overrides w.n): K = V for grad_hidden (plus up to
    ceil(V/256) chunk additions), K = N for grad_weight."""
    tol = TOL[w.dtype]
    n = w.n if n_rows is None else n_rows
    return {"grad_hidden": kappa(tol, w.v, math.ceil(w.v / 256)),
            "grad_weight": kappa(tol, n),
            "grad_bias": bias_kappa(n)}


def to_dev(x: dict) -> dict:
    return {k: (None if t is None else t.cuda()) for k, t in x.items()}


def run_gpu(xd: dict, w, grad_out=1.0, row_metrics=True, vocab_chunk=0,
            grad_weight_dtype=None, backward=True, skip_ignored=False):
    """Forward (+ backward) through the C ABI; returns CPU tensors."""
    err = torch.zeros((), dtype=torch.int32, device="cuda")
    f = api.flce_forward_tensors(xd["hidden"], xd["weight"], xd["targets"], xd["bias"],
                                 w.ignore_index, w.logit_scale, w.softcap, w.reduction,
                                 return_metrics=True, row_metrics=row_metrics, err_word=err,
                                 skip_ignored=skip_ignored, label_smoothing=w.label_smoothing,
                                 z_loss=w.z_loss)
    out = {k: (None if t is None else t.detach().cpu()) for k, t in f.items()}
    if backward:
        if w.reduction == "none":
            go = torch.as_tensor(grad_out, dtype=torch.float32).cuda()
        else:
            go = torch.tensor(float(grad_out), dtype=torch.float32, device="cuda")
        gh, gw, gb = api.flce_backward_tensors(
            xd["hidden"], xd["weight"], xd["targets"], f["lse_rows"], f["n_valid"], go,
            xd["bias"], w.ignore_index, w.logit_scale, w.softcap, w.reduction,
            grad_weight_dtype=grad_weight_dtype, err_word=err, vocab_chunk=vocab_chunk,
            skip_ignored=skip_ignored, label_smoothing=w.label_smoothing, z_loss=w.z_loss)
        out["grad_hidden"] = gh.cpu()
        out["grad_weight"] = gw.cpu()
        out["grad_bias"] = None if gb is None else gb.cpu()
    torch.cuda.synchronize()
    out["err_word"] = int(err.item())
    return out


def oracle_args(x: dict, w):
    return (x["hidden"], x["weight"], x["targets"], x["bias"], w.ignore_index,
            w.logit_scale, w.softcap, w.reduction)


def oracle_opts(w) -> dict:
    return dict(label_smoothing=w.label_smoothing, z_loss=w.z_loss)


def assert_rows_close(name, got, ref, rel, valid=None, floor=None):
    """|got - ref| <= rel |ref| + floor on the rows (of ``valid``)."""
    got = got.to(torch.float64)
    ref = ref.to(torch.float64)
    fl = torch.zeros_like(ref) if floor is None else floor.to(torch.float64)
    if valid is not None:
        got, ref, fl = got[valid], ref[valid], fl[valid]
    err = (got - ref).abs()
    bound = rel * ref.abs() + fl
    bad = ~(err <= bound)
    assert not bool(bad.any()), (
        f"{name}: {int(bad.sum())} of {bad.numel()} rows off; worst abs err "
        f"{float(err.max()):.3e} (rel bound {rel}, worst excess "
        f"{float((err - bound).max()):.3e})")


def assert_scalar_close(name, got: float, ref: float, rel, row_floor_sum=0.0, abs_sum=0.0,
                        n=1):
    """A reduced loss: rel |ref| plus the rows' floors (summed, or averaged by
    the caller) plus the fp32 tree sum's own rounding over n terms whose
    absolute values sum to ``abs_sum``."""
    if math.isnan(ref):
        assert math.isnan(got), (name, got, ref)
        return
    bound = rel * abs(ref) + row_floor_sum + (math.ceil(math.log2(max(n, 2))) + 1) * U24 * abs_sum
    assert abs(got - ref) <= bound, f"{name}: {got} vs {ref} (bound {bound:.3e})"


def assert_grad_close(name, got, ref, tol, mag=None, kap=0.0):
    """Elementwise |got - ref| <= atol + rtol |ref| + g_floor + kap * mag, and
    the normwise bar (see the module docstring)."""
    got = got.to(torch.float64)
    ref = ref.to(torch.float64)
    diff = (got - ref).abs()
    floor = tol.get("g_floor", 0.0)  # output-format floor, see TOL["f16"]
    bound = tol["g_atol"] + tol["g_rtol"] * ref.abs() + floor
    if mag is not None:
        bound = bound + kap * mag.to(torch.float64)
    bad = ~(diff <= bound)
    assert not bool(bad.any()), (
        f"{name}: {int(bad.sum())} of {bad.numel()} entries beyond the elementwise bar; "
        f"worst err {float(diff.max()):.3e}, worst excess {float((diff - bound).max()):.3e}")
    rn = float(ref.norm())
    dn = float((got - ref).norm())
    if rn > 0:
        nb = tol["g_norm"] * rn + floor * math.sqrt(ref.numel())
        assert dn <= nb, f"{name}: normwise rel err {dn / rn:.3e} > {tol['g_norm']} (+ floor)"
    else:
        assert dn <= tol["g_atol"] * math.sqrt(max(1, ref.numel())), f"{name}: expected zeros"


def check_forward(out, ref, w, tol, skipped=False):
    """``skipped``: ignored rows were left out of the contractions, so their
    lse and entropy are not computed (NaN) and only valid rows are compared."""
    nv = ref["n_valid"]
    assert int(out["n_valid"]) == nv
    valid = ref["valid"]
    floor = row_floor(w.h, ce_row_ops(ref))
    assert_rows_close("loss_rows", out["loss_rows"], ref["loss"], tol["loss_rel"], floor=floor)
    stat_rows = valid if skipped else None
    assert_rows_close("lse_rows", out["lse_rows"], ref["lse"], tol["loss_rel"], stat_rows,
                      floor=floor)
    if skipped:
        assert bool(torch.isnan(out["lse_rows"][~valid]).all())
    assert torch.all(out["loss_rows"][~valid] == 0)
    if w.reduction != "none":
        fsum = float(floor[valid & torch.isfinite(floor)].sum())
        asum = float(ref["loss"][valid].abs().nan_to_num(0.0).sum())
        if w.reduction == "mean" and nv > 0:
            fsum, asum = fsum / nv, asum / nv
        assert_scalar_close("loss", float(out["loss"]), float(ref["loss_out"]), tol["loss_rel"],
                            fsum, asum, max(nv, 1))
    # argmax-based correctness where the top-2 gap is decisive; on near-tie
    # rows either answer can be right, but a row reported correct must have
    # its target logit within the tie window of the row maximum
    decisive = ref["top2_gap"] > 1e-2
    corr = out["correct_rows"].bool()
    assert torch.equal(corr[decisive], ref["correct"][decisive]), "correct_rows differ"
    near = ~decisive & valid & corr
    if bool(near.any()):
        slack = (ref["max_logit"] - ref["target_logit"])[near]
        assert bool((slack <= 1e-2).all()), f"near-tie row reported correct off the tie: {slack}"
    assert_rows_close("entropy_rows", out["entropy_rows"], ref["entropy"], tol["ent_rel"],
                      stat_rows, floor=floor)
    if nv > 0:
        acc_ref = ref["mean_token_accuracy"]
        # rows with a near-tie may legitimately resolve either way
        slack = int((~decisive & valid).sum()) / nv
        assert abs(float(out["metrics"][0]) - acc_ref) <= slack + 1e-6
        ent_floor = float(floor[valid].sum()) / nv
        assert_scalar_close("entropy", float(out["metrics"][1]), ref["entropy_mean"],
                            tol["ent_rel"], ent_floor, float(ref["entropy"][valid].abs().sum()) / nv,
                            nv)


def check_backward(out, gref, tol, has_bias, kappas):
    """Gradients against an oracle backward run with magnitudes=True;
    ``kappas`` from grad_kappas()."""
    for k in ("grad_hidden", "grad_weight") + (("grad_bias",) if has_bias else ()):
        assert_grad_close(k, out[k], gref[k], tol, gref[k + "_mag"], kappas[k])
