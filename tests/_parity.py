"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 oracle on the same seeded inputs.

Tolerances (GPU vs oracle):
  * loss and lse per row: rel 1e-5 for fp32 inputs, 2e-3 for bf16 inputs;
  * gradients elementwise: |d| <= atol + rtol*|ref| with (5e-5, 5e-2) for
    bf16 and (1e-5, 1e-4) for fp32. These bars are stated for the gradient of
    a mean-reduced loss; the gradient of a 'sum' loss (and of 'none' with
    per-row upstream gradients of order 1) is n_valid times larger, so for
    those reductions both sides are divided by n_valid before the
    elementwise test (rtol is scale-free and unchanged);
  * fp16 outputs: both gradient bars widen by the half-spacing of fp16
    subnormals (2^-25, unscaled), the error of storing a gradient below
    fp16's smallest normal value whatever the kernel computes;
  * gradients normwise: ||d|| / ||ref|| <= 1e-2 for bf16 (D is rounded to
    bf16, relative error 2^-9 per element, and the outputs to bf16) and
    1e-4 for fp32. The elementwise bar alone passes anything when gradients
    are ~1e-6 (a mean over thousands of rows), so the normwise bar is what
    catches a wrong factor or index there;
  * argmax-based correctness: bit-exact on rows whose top-2 logit gap in the
    oracle exceeds 1e-2;
  * entropy per row: rel 1e-3 (bf16) / 1e-4 (fp32).
"""
from __future__ import annotations

import math

import torch

import oracle
from linear_cross_entropy_vocab_gb300 import api

TOL = {
    "f32": dict(loss_rel=1e-5, g_atol=1e-5, g_rtol=1e-4, g_norm=1e-4, ent_rel=1e-4),
    "bf16": dict(loss_rel=2e-3, g_atol=5e-5, g_rtol=5e-2, g_norm=1e-2, ent_rel=1e-3),
}
# fp16 inputs: the pages state no fp16 bar. fp16 rounds more finely than bf16
# (2^-11 against 2^-8 relative) in every place the bf16 path rounds (D and the
# outputs), so the bf16 bars bound the fp16 path, except where fp16's narrow
# exponent range bites: gradients stored in fp16 below its smallest normal
# value (2^-14) are subnormal, spaced 2^-24 apart, so rounding an output there
# errs by up to 2^-25 absolute whatever the kernel does (a 'mean' KL divergence
# divides by N*V and lands there). ``g_floor`` adds that half-spacing, on the
# unscaled output, to the elementwise and normwise bars.
TOL["f16"] = dict(TOL["bf16"], g_floor=2.0 ** -25)


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


def assert_rows_close(name, got, ref, rel, valid=None):
    got = got.to(torch.float64)
    ref = ref.to(torch.float64)
    if valid is not None:
        got, ref = got[valid], ref[valid]
    err = (got - ref).abs()
    bound = rel * ref.abs().clamp_min(1.0)
    bad = err > bound
    assert not bool(bad.any()), (
        f"{name}: {int(bad.sum())} of {bad.numel()} rows off; worst abs err "
        f"{float(err.max()):.3e} (rel bound {rel})")


def assert_grad_close(name, got, ref, tol, scale=1.0):
    got = got.to(torch.float64) * scale
    ref = ref.to(torch.float64) * scale
    diff = (got - ref).abs()
    floor = tol.get("g_floor", 0.0) * abs(scale)  # output-format floor, see TOL["f16"]
    bound = tol["g_atol"] + tol["g_rtol"] * ref.abs() + floor
    bad = diff > bound
    assert not bool(bad.any()), (
        f"{name}: {int(bad.sum())} of {bad.numel()} entries beyond atol+rtol; worst "
        f"{float(diff.max()):.3e}")
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
    assert_rows_close("loss_rows", out["loss_rows"], ref["loss"], tol["loss_rel"])
    stat_rows = valid if skipped else None
    assert_rows_close("lse_rows", out["lse_rows"], ref["lse"], tol["loss_rel"], stat_rows)
    if skipped:
        assert bool(torch.isnan(out["lse_rows"][~valid]).all())
    assert torch.all(out["loss_rows"][~valid] == 0)
    if w.reduction != "none":
        r = ref["loss_out"]
        g = float(out["loss"])
        if math.isnan(r):
            assert math.isnan(g)
        else:
            assert abs(g - r) <= tol["loss_rel"] * max(1.0, abs(r)), (g, r)
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
                      stat_rows)
    if nv > 0:
        acc_ref = ref["mean_token_accuracy"]
        # rows with a near-tie may legitimately resolve either way
        slack = int((~decisive & valid).sum()) / nv
        assert abs(float(out["metrics"][0]) - acc_ref) <= slack + 1e-6
        assert abs(float(out["metrics"][1]) - ref["entropy_mean"]) <= tol["ent_rel"] * max(
            1.0, abs(ref["entropy_mean"]))


def grad_scale(reduction: str, n_valid: int) -> float:
    """Factor that brings a gradient to the scale of the mean-reduced loss."""
    if reduction == "mean" or n_valid == 0:
        return 1.0
    return 1.0 / n_valid


def check_backward(out, gref, tol, has_bias, scale=1.0):
    assert_grad_close("grad_hidden", out["grad_hidden"], gref["grad_hidden"], tol, scale)
    assert_grad_close("grad_weight", out["grad_weight"], gref["grad_weight"], tol, scale)
    if has_bias:
        assert_grad_close("grad_bias", out["grad_bias"], gref["grad_bias"], tol, scale)
