"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against a fact the kernel card or the mathematics
fixes: a pure-Python brute force with explicit softmax, central finite
differences of the loss, closed forms (W=0, V=1, a dominant logit), the
posterior-mass identity, ignored-row and reduction invariants, and the torch
library's own cross_entropy with autograd. ``test_planted_mistakes`` plants a
set of plausible mistakes in the oracle and shows that these pins catch every
one of them.

Definitions followed: "fused-linear-ce" (trl-lib model card) §Full signature,
§Metrics for free, §Algorithm.
"""
import math

import pytest
import torch

import oracle
from oracle import brute, flce_oracle
from linear_cross_entropy_vocab_gb300.workloads import Workload, make_inputs

F64 = torch.float64

CASES = [
    # name, n, h, v, bias, softcap, scale, ignore_frac, reduction
    ("plain", 9, 6, 13, False, None, 1.0, 0.0, "mean"),
    ("bias_ignore", 12, 5, 17, True, None, 1.0, 0.25, "mean"),
    ("softcap_scale", 10, 7, 11, True, 1.5, 0.6, 0.2, "sum"),
    ("none_reduction", 8, 4, 9, False, 2.0, 1.3, 0.25, "none"),
    ("scale_only", 7, 8, 23, True, None, 2.5, 0.0, "sum"),
]


def _inputs(n, h, v, bias, softcap, scale, ignore_frac, reduction, seed=0,
            hidden_var=1.0):
    w = Workload("pin", n, h, v, "f32", hidden_var=hidden_var,
                 weight_var=1.0 / h,
                 bias_var=0.5 if bias else None, ignore_frac=ignore_frac,
                 logit_scale=scale, softcap=softcap, reduction=reduction,
                 seed=seed)
    x = make_inputs(w)
    return {k: (None if t is None else (t.to(F64) if t.is_floating_point() else t))
            for k, t in x.items()}


def _opts(case):
    _, n, h, v, bias, softcap, scale, frac, red = case
    return dict(logit_scale=scale, softcap=softcap, reduction=red)


def _lists(x):
    b = None if x["bias"] is None else x["bias"].tolist()
    return x["hidden"].tolist(), x["weight"].tolist(), x["targets"].tolist(), b


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_brute_force_forward(case):
    x = _inputs(*case[1:])
    o = _opts(case)
    f = oracle.forward(x["hidden"], x["weight"], x["targets"], x["bias"], -100,
                       o["logit_scale"], o["softcap"], o["reduction"])
    h, w, t, b = _lists(x)
    rows = brute.per_row(h, w, t, b, -100, o["logit_scale"], o["softcap"])
    for i, r in enumerate(rows):
        assert f["loss"][i].item() == pytest.approx(r["loss"], rel=1e-12, abs=1e-14)
        assert f["entropy"][i].item() == pytest.approx(r["entropy"], rel=1e-12)
        assert int(f["argmax"][i]) == r["argmax"]
        assert bool(f["correct"][i]) == r["correct"]
    ref = brute.loss(h, w, t, b, -100, o["logit_scale"], o["softcap"], o["reduction"])
    if o["reduction"] == "none":
        assert torch.allclose(f["loss_out"], torch.tensor(ref, dtype=F64), rtol=1e-12)
    else:
        assert f["loss_out"] == pytest.approx(ref, rel=1e-12)
    acc, ent = brute.metrics(h, w, t, b, -100, o["logit_scale"], o["softcap"])
    assert f["mean_token_accuracy"] == pytest.approx(acc, rel=1e-15)
    assert f["entropy_mean"] == pytest.approx(ent, rel=1e-12)


def _fd_check(case, n_probe=6, step=1e-5, seed=1, mod=flce_oracle, label_smoothing=0.0,
              z_loss=0.0):
    """Central differences of the brute-force loss against the oracle's
    analytic gradients, at randomly chosen entries of hidden, weight, bias."""
    x = _inputs(*case[1:])
    o = _opts(case)
    n = x["hidden"].shape[0]
    gen = torch.Generator().manual_seed(seed)
    row_g = None
    grad_out = 0.7
    if o["reduction"] == "none":
        row_g = (torch.rand(n, generator=gen, dtype=F64) + 0.5)
        grad_out = row_g
    g = mod.backward(x["hidden"], x["weight"], x["targets"], x["bias"], -100,
                     o["logit_scale"], o["softcap"], o["reduction"], grad_out,
                     label_smoothing=label_smoothing, z_loss=z_loss)
    scale = 1.0 if o["reduction"] == "none" else 0.7

    def L(hh, ww, bb):
        b = None if bb is None else bb.tolist()
        val = brute.loss(hh.tolist(), ww.tolist(), x["targets"].tolist(), b, -100,
                         o["logit_scale"], o["softcap"], o["reduction"],
                         None if row_g is None else row_g.tolist(),
                         label_smoothing=label_smoothing, z_loss=z_loss)
        return scale * val

    worst = 0.0
    for name, key in (("hidden", "grad_hidden"), ("weight", "grad_weight"),
                      ("bias", "grad_bias")):
        if x[name] is None:
            continue
        base = x[name]
        for _ in range(n_probe):
            flat = int(torch.randint(0, base.numel(), (1,), generator=gen))
            plus = base.clone().reshape(-1)
            minus = base.clone().reshape(-1)
            plus[flat] += step
            minus[flat] -= step
            args = {"hidden": x["hidden"], "weight": x["weight"], "bias": x["bias"]}
            args[name] = plus.reshape(base.shape)
            lp = L(args["hidden"], args["weight"], args["bias"])
            args[name] = minus.reshape(base.shape)
            lm = L(args["hidden"], args["weight"], args["bias"])
            fd = (lp - lm) / (2 * step)
            an = g[key].reshape(-1)[flat].item()
            err = abs(fd - an) / max(1e-6, abs(an), abs(fd))
            worst = max(worst, err)
    return worst


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_finite_differences(case):
    assert _fd_check(case) < 1e-6


# label smoothing / z-loss: (case, eps, lam)
OPT_CASES = [
    (CASES[1], 0.1, 0.0),
    (CASES[2], 0.0, 1e-2),
    (CASES[3], 0.2, 5e-3),
    (CASES[4], 0.05, 1e-3),
]


@pytest.mark.parametrize("case,eps,lam", OPT_CASES, ids=[f"{c[0]}-ls{e}-z{z}" for c, e, z in OPT_CASES])
def test_smoothing_zloss_brute_force_and_fd(case, eps, lam):
    """Label smoothing and z-loss: the oracle's per-row loss against the brute
    force's cross-entropy against (1-eps)*onehot + eps/V plus lam*lse^2, and
    its gradients against central differences of that brute-force loss."""
    x = _inputs(*case[1:])
    o = _opts(case)
    f = oracle.forward(x["hidden"], x["weight"], x["targets"], x["bias"], -100,
                       o["logit_scale"], o["softcap"], o["reduction"],
                       label_smoothing=eps, z_loss=lam)
    h, w, t, b = _lists(x)
    rows = brute.per_row(h, w, t, b, -100, o["logit_scale"], o["softcap"], eps, lam)
    for i, r in enumerate(rows):
        assert f["loss"][i].item() == pytest.approx(r["loss"], rel=1e-12, abs=1e-14)
    assert _fd_check(case, label_smoothing=eps, z_loss=lam) < 1e-6


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_torch_label_smoothing_and_zloss(reduction):
    """Library cross-check of label smoothing: torch cross_entropy with
    label_smoothing (its own ignore_index handling) plus the z-loss term, with
    autograd for the gradients."""
    eps, lam = 0.15, 2e-3
    x = _inputs(16, 8, 27, True, 2.5, 0.7, 0.25, reduction)
    hid = x["hidden"].clone().requires_grad_(True)
    wt = x["weight"].clone().requires_grad_(True)
    bs = x["bias"].clone().requires_grad_(True)
    logits = 2.5 * torch.tanh(0.7 * torch.nn.functional.linear(hid, wt, bs) / 2.5)
    ce = torch.nn.functional.cross_entropy(logits, x["targets"], ignore_index=-100,
                                           reduction="none", label_smoothing=eps)
    valid = (x["targets"] != -100).to(F64)
    rows = ce + lam * torch.logsumexp(logits, dim=1) ** 2 * valid
    if reduction == "mean":
        ref = rows.sum() / valid.sum()
    elif reduction == "sum":
        ref = rows.sum()
    else:
        ref = rows
    gen = torch.Generator().manual_seed(3)
    go = torch.rand(16, generator=gen, dtype=F64) if reduction == "none" else 1.0
    (ref * go).sum().backward() if reduction == "none" else ref.backward()
    args = (x["hidden"], x["weight"], x["targets"], x["bias"], -100, 0.7, 2.5, reduction)
    f = oracle.forward(*args, label_smoothing=eps, z_loss=lam)
    if reduction == "none":
        assert torch.allclose(f["loss_out"], ref.detach(), rtol=1e-12, atol=1e-14)
    else:
        assert f["loss_out"] == pytest.approx(ref.item(), rel=1e-12)
    g = oracle.backward(*args, go, label_smoothing=eps, z_loss=lam)
    assert torch.allclose(g["grad_hidden"], hid.grad, rtol=1e-11, atol=1e-15)
    assert torch.allclose(g["grad_weight"], wt.grad, rtol=1e-11, atol=1e-15)
    assert torch.allclose(g["grad_bias"], bs.grad, rtol=1e-11, atol=1e-15)


def test_closed_form_zero_weight_with_options():
    """W = 0, b = 0: lse = ln V and every logit is 0, so with any label
    smoothing the loss is ln V, plus lam * (ln V)^2 from the z-loss."""
    n, h, v = 9, 5, 41
    x = _inputs(n, h, v, False, None, 1.0, 0.0, "mean")
    w0 = torch.zeros(v, h, dtype=F64)
    for eps, lam in ((0.3, 0.0), (0.0, 0.01), (0.1, 0.02)):
        f = oracle.forward(x["hidden"], w0, x["targets"], None, -100, 1.0, None, "mean",
                           label_smoothing=eps, z_loss=lam)
        lnv = math.log(v)
        assert f["loss_out"] == pytest.approx(lnv + lam * lnv * lnv, rel=1e-14)


def test_closed_form_zero_weight():
    """W = 0, b = 0: every logit is 0, so p = 1/V, loss_i = ln V, entropy =
    ln V, argmax = 0, grad_hidden = 0 and grad_weight_j = g * sum_i (1/V -
    [t_i = j]) h_i."""
    n, h, v = 11, 6, 37
    x = _inputs(n, h, v, False, None, 1.0, 0.2, "mean")
    w0 = torch.zeros(v, h, dtype=F64)
    b0 = torch.zeros(v, dtype=F64)
    f = oracle.forward(x["hidden"], w0, x["targets"], b0, -100, 1.0, None, "mean")
    valid = x["targets"] != -100
    lnv = math.log(v)
    assert torch.allclose(f["lse"], torch.full((n,), lnv, dtype=F64), rtol=0, atol=1e-14)
    assert torch.allclose(f["loss"][valid], torch.full((int(valid.sum()),), lnv, dtype=F64),
                          rtol=0, atol=1e-14)
    assert f["loss_out"] == pytest.approx(lnv, abs=1e-14)
    assert f["entropy_mean"] == pytest.approx(lnv, abs=1e-13)
    assert (f["argmax"] == 0).all()
    g = oracle.backward(x["hidden"], w0, x["targets"], b0, -100, 1.0, None, "mean", 1.0)
    assert torch.equal(g["grad_hidden"], torch.zeros(n, h, dtype=F64))
    nv = int(valid.sum())
    exp_gw = torch.zeros(v, h, dtype=F64)
    exp_gb = torch.zeros(v, dtype=F64)
    for i in range(n):
        ti = int(x["targets"][i])
        if ti == -100:
            continue
        for j in range(v):
            c = (1.0 / v - (1.0 if j == ti else 0.0)) / nv
            exp_gw[j] += c * x["hidden"][i]
            exp_gb[j] += c
    assert torch.allclose(g["grad_weight"], exp_gw, rtol=1e-12, atol=1e-15)
    assert torch.allclose(g["grad_bias"], exp_gb, rtol=1e-12, atol=1e-15)


def test_closed_form_bias_only_softcap():
    """W = 0 with a bias: z_j = c*tanh(s*b_j/c) for every row, so each row's
    loss is log(sum_j e^{z_j}) - z_{t_i}, independent of the hidden state."""
    n, h, v = 7, 5, 19
    x = _inputs(n, h, v, True, 3.0, 0.8, 0.0, "none")
    w0 = torch.zeros(v, h, dtype=F64)
    f = oracle.forward(x["hidden"], w0, x["targets"], x["bias"], -100, 0.8, 3.0, "none")
    z = [3.0 * math.tanh(0.8 * float(b) / 3.0) for b in x["bias"]]
    lse = math.log(math.fsum(math.exp(q) for q in z))
    for i in range(n):
        assert f["loss"][i].item() == pytest.approx(lse - z[int(x["targets"][i])], rel=1e-13)


def test_vocab_of_one():
    """V = 1: p = 1 = onehot, so the loss and all gradients are 0."""
    x = _inputs(6, 4, 1, True, None, 1.0, 0.0, "sum")
    f = oracle.forward(x["hidden"], x["weight"], x["targets"], x["bias"], -100, 1.0, None, "sum")
    assert f["loss_out"] == 0.0
    g = oracle.backward(x["hidden"], x["weight"], x["targets"], x["bias"], -100, 1.0, None, "sum", 1.0)
    assert torch.all(g["grad_hidden"].abs() < 1e-15)
    assert torch.all(g["grad_weight"].abs() < 1e-15)
    assert torch.all(g["grad_bias"].abs() < 1e-15)


@pytest.mark.parametrize("gap", [50.0, 10.0])
def test_dominant_logit(gap):
    """A logit ``gap`` above all others (the logit=50 peaked rows of the
    CuTe-DSL CE PR's tolerance note): loss = log(1 + (V-1) e^{-gap}),
    argmax = target. At gap 50 the exact loss (~3e-21) is below the fp64
    resolution of lse (~50 * 2^-52), so it is checked in absolute terms."""
    v = 16
    t = torch.arange(8) * 2 % v
    hidden = gap * torch.nn.functional.one_hot(t, v).to(F64)
    weight = torch.eye(v, dtype=F64)
    f = oracle.forward(hidden, weight, t, None, -100, 1.0, None, "none")
    expect = math.log1p((v - 1) * math.exp(-gap))
    full = torch.full((8,), expect, dtype=F64)
    if gap >= 40:
        assert torch.allclose(f["loss"], full, rtol=0, atol=1e-13)
    else:
        assert torch.allclose(f["loss"], full, rtol=1e-9, atol=0)
    assert (f["argmax"] == t).all()
    assert f["mean_token_accuracy"] == 1.0
    assert f["top2_gap"].eq(gap).all()


@pytest.mark.parametrize("scale", [1.0])
def test_posterior_mass_identity(scale):
    """Softcap off, logit_scale 1: sum_j (p_ij - onehot_ij) = 0 for every row,
    hence sum_j grad_bias_j = 0 and sum_j grad_weight_j = 0."""
    x = _inputs(13, 6, 29, True, None, scale, 0.2, "sum")
    g = oracle.backward(x["hidden"], x["weight"], x["targets"], x["bias"], -100, scale, None, "sum", 1.0)
    assert abs(float(g["grad_bias"].sum())) < 1e-13
    assert g["grad_weight"].sum(dim=0).abs().max() < 1e-13


def test_ignored_rows_contribute_nothing():
    """Ignored rows: zero loss, an exactly zero grad_hidden row, and their
    hidden state has no effect on the loss, grad_weight or grad_bias."""
    x = _inputs(12, 5, 21, True, 4.0, 0.9, 0.34, "mean")
    ign = (x["targets"] == -100)
    assert int(ign.sum()) == 4
    f = oracle.forward(x["hidden"], x["weight"], x["targets"], x["bias"], -100, 0.9, 4.0, "mean")
    assert torch.all(f["loss"][ign] == 0)
    g = oracle.backward(x["hidden"], x["weight"], x["targets"], x["bias"], -100, 0.9, 4.0, "mean", 1.0)
    assert torch.all(g["grad_hidden"][ign] == 0)
    h2 = x["hidden"].clone()
    h2[ign] = 123.0
    f2 = oracle.forward(h2, x["weight"], x["targets"], x["bias"], -100, 0.9, 4.0, "mean")
    g2 = oracle.backward(h2, x["weight"], x["targets"], x["bias"], -100, 0.9, 4.0, "mean", 1.0)
    assert f2["loss_out"] == pytest.approx(f["loss_out"], rel=1e-14)
    assert torch.allclose(g2["grad_weight"], g["grad_weight"], rtol=1e-12, atol=1e-16)
    assert torch.allclose(g2["grad_bias"], g["grad_bias"], rtol=1e-12, atol=1e-16)


def test_reduction_relations():
    x = _inputs(20, 6, 31, True, 5.0, 1.1, 0.15, "mean")
    args = (x["hidden"], x["weight"], x["targets"], x["bias"], -100, 1.1, 5.0)
    fm = oracle.forward(*args, "mean")
    fs = oracle.forward(*args, "sum")
    fn = oracle.forward(*args, "none")
    nv = fm["n_valid"]
    assert nv == 20 - 3
    assert fs["loss_out"] == pytest.approx(fm["loss_out"] * nv, rel=1e-14)
    assert float(fn["loss_out"].sum()) == pytest.approx(fs["loss_out"], rel=1e-14)
    # per-row upstream gradient of 1/n_valid on each row equals 'mean'
    gm = oracle.backward(*args, "mean", 1.0)
    gn = oracle.backward(*args, "none", torch.full((20,), 1.0 / nv, dtype=F64))
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        assert torch.allclose(gm[k], gn[k], rtol=1e-13, atol=1e-17)


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("softcap,scale", [(None, 1.0), (2.5, 0.7)])
def test_torch_library_cross_entropy(reduction, softcap, scale):
    """Library cross-check: torch.nn.functional.cross_entropy on fp64 logits
    (with its own ignore_index handling) and autograd for the gradients."""
    x = _inputs(16, 8, 27, True, softcap, scale, 0.25, reduction)
    hid = x["hidden"].clone().requires_grad_(True)
    wt = x["weight"].clone().requires_grad_(True)
    bs = x["bias"].clone().requires_grad_(True)
    logits = scale * torch.nn.functional.linear(hid, wt, bs)
    if softcap:
        logits = softcap * torch.tanh(logits / softcap)
    ref = torch.nn.functional.cross_entropy(logits, x["targets"], ignore_index=-100,
                                            reduction=reduction)
    gen = torch.Generator().manual_seed(3)
    if reduction == "none":
        go = torch.rand(16, generator=gen, dtype=F64)
        (ref * go).sum().backward()
    else:
        go = 1.0
        ref.backward()
    f = oracle.forward(x["hidden"], x["weight"], x["targets"], x["bias"], -100, scale, softcap, reduction)
    if reduction == "none":
        assert torch.allclose(f["loss_out"], ref.detach(), rtol=1e-12, atol=1e-14)
    else:
        assert f["loss_out"] == pytest.approx(ref.item(), rel=1e-12)
    g = oracle.backward(x["hidden"], x["weight"], x["targets"], x["bias"], -100, scale, softcap, reduction, go)
    assert torch.allclose(g["grad_hidden"], hid.grad, rtol=1e-11, atol=1e-15)
    assert torch.allclose(g["grad_weight"], wt.grad, rtol=1e-11, atol=1e-15)
    assert torch.allclose(g["grad_bias"], bs.grad, rtol=1e-11, atol=1e-15)
    # argmax of the library logits, lowest index on ties
    assert torch.equal(f["argmax"], torch.argmax(logits.detach(), dim=1))


def test_no_valid_rows():
    """n_valid = 0: 'mean' gives NaN loss and metrics, every gradient is 0;
    'sum' gives 0."""
    x = _inputs(5, 4, 9, True, None, 1.0, 0.0, "mean")
    t = torch.full((5,), -100, dtype=torch.int64)
    f = oracle.forward(x["hidden"], x["weight"], t, x["bias"], -100, 1.0, None, "mean")
    assert math.isnan(f["loss_out"]) and math.isnan(f["mean_token_accuracy"])
    assert math.isnan(f["entropy_mean"])
    assert oracle.forward(x["hidden"], x["weight"], t, x["bias"], -100, 1.0, None, "sum")["loss_out"] == 0.0
    g = oracle.backward(x["hidden"], x["weight"], t, x["bias"], -100, 1.0, None, "mean", 1.0)
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        assert torch.count_nonzero(g[k]) == 0


def test_target_out_of_range():
    """A target outside [0, V) that is not ignore_index: flagged, NaN row
    loss, counted in n_valid, never correct, no gradient contribution."""
    x = _inputs(6, 4, 9, False, None, 1.0, 0.0, "sum")
    t = x["targets"].clone()
    t[2] = 9
    t[4] = -3
    f = oracle.forward(x["hidden"], x["weight"], t, None, -100, 1.0, None, "sum")
    assert f["target_error"]
    assert f["n_valid"] == 6
    assert math.isnan(f["loss"][2]) and math.isnan(f["loss"][4])
    assert not f["correct"][2] and not f["correct"][4]
    g = oracle.backward(x["hidden"], x["weight"], t, None, -100, 1.0, None, "sum", 1.0)
    assert torch.count_nonzero(g["grad_hidden"][2]) == 0
    assert torch.count_nonzero(g["grad_hidden"][4]) == 0


def test_sampled_rows_match_full():
    """The sampled interfaces used at full size agree with the full pass."""
    x = _inputs(40, 6, 50, True, 3.0, 0.8, 0.1, "mean")
    args = (x["hidden"], x["weight"], x["targets"], x["bias"], -100, 0.8, 3.0, "mean")
    full = oracle.forward(*args)
    rows = [0, 7, 39, 12]
    part = oracle.forward(*args, rows=rows)
    for k in ("loss", "lse", "entropy", "argmax", "top2_gap"):
        assert torch.equal(part[k], full[k][rows])
    g_full = oracle.backward(*args, 1.0)
    vr = [0, 49, 17, 3]
    g_part = oracle.backward(*args, 1.0, lse=full["lse"], rows=rows, vocab_rows=vr)
    assert torch.allclose(g_part["grad_hidden"], g_full["grad_hidden"][rows], rtol=1e-13, atol=1e-18)
    assert torch.allclose(g_part["grad_weight"], g_full["grad_weight"][vr], rtol=1e-13, atol=1e-18)
    assert torch.allclose(g_part["grad_bias"], g_full["grad_bias"][vr], rtol=1e-13, atol=1e-18)


# ---------------------------------------------------------------------------
# Planted mistakes: each mutant must be caught by at least one pin.

def _mut_drop_bias(h, w, b, s, c):
    return flce_oracle_orig_final_logits(h, w, None, s, c)


def _mut_scale_after_cap(h, w, b, s, c):
    lin = h.to(F64) @ w.to(F64).T
    if b is not None:
        lin = lin + b.to(F64)
    z = c * torch.tanh(lin / c) if c else lin
    return s * z, s * lin


def _mut_transposed(h, w, b, s, c):
    # uses the wrong weight rows: W reversed along the vocabulary
    return flce_oracle_orig_final_logits(h, torch.flip(w, [0]), b, s, c)


def _mut_dlogits_no_cap(z, u, lse, pos, g, s, c, *opts):
    return flce_oracle_orig_dlogits(z, u, lse, pos, g, s, None, *opts)


def _mut_dlogits_sign(z, u, lse, pos, g, s, c, *opts):
    return -flce_oracle_orig_dlogits(z, u, lse, pos, g, s, c, *opts)


def _mut_dlogits_no_onehot(z, u, lse, pos, g, s, c, *opts):
    return flce_oracle_orig_dlogits(z, u, lse, torch.full_like(pos, -1), g, s, c, *opts)


def _mut_dlogits_no_scale(z, u, lse, pos, g, s, c, *opts):
    return flce_oracle_orig_dlogits(z, u, lse, pos, g, 1.0, c, *opts)


def _mut_dlogits_no_zloss_term(z, u, lse, pos, g, s, c, eps=0.0, lam=0.0, v=0):
    return flce_oracle_orig_dlogits(z, u, lse, pos, g, s, c, eps, 0.0, v)


def _mut_dlogits_no_uniform_term(z, u, lse, pos, g, s, c, eps=0.0, lam=0.0, v=0):
    d = flce_oracle_orig_dlogits(z, u, lse, pos, g, s, c, eps, lam, v)
    return d + (eps / v) * g[:, None] * s if v else d


def _mut_dlogits_full_onehot(z, u, lse, pos, g, s, c, eps=0.0, lam=0.0, v=0):
    # uses 1 instead of 1 - eps on the target
    d = flce_oracle_orig_dlogits(z, u, lse, pos, g, s, c, eps, lam, v)
    hit = pos >= 0
    d[torch.nonzero(hit).flatten(), pos[hit]] -= eps * g[hit] * s
    return d


flce_oracle_orig_final_logits = flce_oracle.final_logits
flce_oracle_orig_dlogits = flce_oracle._dlogits

MUTANTS = [
    ("final_logits", _mut_drop_bias),
    ("final_logits", _mut_scale_after_cap),
    ("final_logits", _mut_transposed),
    ("_dlogits", _mut_dlogits_no_cap),
    ("_dlogits", _mut_dlogits_sign),
    ("_dlogits", _mut_dlogits_no_onehot),
    ("_dlogits", _mut_dlogits_no_scale),
    ("_dlogits", _mut_dlogits_no_zloss_term),
    ("_dlogits", _mut_dlogits_no_uniform_term),
    ("_dlogits", _mut_dlogits_full_onehot),
]


def _pins_pass():
    try:
        for case in CASES:
            test_brute_force_forward(case)
            if _fd_check(case, n_probe=3) >= 1e-6:
                return False
        for case, eps, lam in OPT_CASES:
            if _fd_check(case, n_probe=3, label_smoothing=eps, z_loss=lam) >= 1e-6:
                return False
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("target,mutant", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_planted_mistakes(monkeypatch, target, mutant):
    assert _pins_pass()  # the unmodified oracle passes
    monkeypatch.setattr(flce_oracle, target, mutant)
    assert not _pins_pass(), f"planted mistake {mutant.__name__} went unnoticed"


def test_max_logit_and_gap_match_brute_force():
    """max_logit and top2_gap, which the GPU tests use to tell decisive argmax
    rows from near-ties, against the brute force's logits."""
    g = torch.Generator().manual_seed(21)
    hid = torch.randn(7, 5, generator=g, dtype=torch.float64)
    w = torch.randn(11, 5, generator=g, dtype=torch.float64)
    b = torch.randn(11, generator=g, dtype=torch.float64) * 0.2
    t = torch.randint(0, 11, (7,), generator=g)
    f = oracle.forward(hid, w, t, b, -100, 0.8, 3.0, "mean")
    z = brute.logits(hid.tolist(), w.tolist(), b.tolist(), 0.8, 3.0)
    for i, row in enumerate(z):
        srt = sorted(row, reverse=True)
        assert f["max_logit"][i].item() == pytest.approx(srt[0], rel=1e-12)
        assert f["top2_gap"][i].item() == pytest.approx(srt[0] - srt[1], rel=1e-9, abs=1e-12)
        assert f["target_logit"][i].item() == pytest.approx(row[int(t[i])], rel=1e-12)
