"""GPU parity of the fused linear KL divergence (FusedLinearKLDivLoss pull
request, Liger-Kernel #1423): the CUDA path through the C ABI against the
fp64 KL oracle, element by element, on seeded inputs with ragged tails along
N, V and H, every reduction, temperature, labels with ignored rows (with and
without leaving them out of the contractions), bias, top-k truncated teachers
(exact zeros, so the eps clamp matters), multi-chunk backward passes, and the
three input dtypes.

Tolerances are those of the cross-entropy (``tests/_parity.py``), in each
output's own units: loss and lse rows rel 2e-3 (16-bit inputs) / 1e-5 (fp32)
plus an fp32 evaluation floor on |lse| Q + |loss - lse Q|; per-row sums of q
rel 1e-5 (a sum of non-negative fp32 terms); gradients atol + rtol plus the
rounding of D times the sum of the absolute terms of each entry, and the
normwise bar.
"""
import math

import pytest
import torch

from _parity import (TOL, assert_grad_close, assert_rows_close, assert_scalar_close,
                     grad_kappas, kl_row_ops, row_floor, to_dev)
from linear_cross_entropy_vocab_gb300 import api, fused_linear_kl_div
from linear_cross_entropy_vocab_gb300.workloads import Workload, make_inputs, make_teacher_probs
from oracle import kl_oracle

pytestmark = pytest.mark.gpu


def _w(name, n, h, v, dtype="bf16", **kw):
    return Workload(name, n, h, v, dtype, **kw)


# (workload, temperature, reduction, with labels, teacher keep_top, vocab_chunk, skip_ignored)
CASES = [
    (_w("tails_bias_bm", 300, 136, 1000, bias_var=0.02, ignore_frac=0.1), 1.0, "batchmean",
     True, None, 0, False),
    (_w("v32003_sum", 512, 256, 32003), 2.0, "sum", False, None, 0, False),
    (_w("n4097_mean", 4097, 512, 4096, ignore_frac=0.1), 0.5, "mean", True, None, 0, False),
    (_w("topk_none_bias", 640, 192, 5000, bias_var=0.02, ignore_frac=0.2), 1.5, "none", True,
     20, 512, False),
    (_w("skip_bm", 300, 136, 1000, bias_var=0.02, ignore_frac=0.3), 1.0, "batchmean", True,
     None, 0, True),
    (_w("skip_none_chunks", 1000, 256, 3000, ignore_frac=0.25), 2.0, "none", True, 50, 512,
     True),
    (_w("f16_bm", 384, 256, 3000, "f16", ignore_frac=0.05), 1.0, "batchmean", True, None, 0,
     False),
    (_w("f16_skip_mean_bias", 500, 128, 2056, "f16", bias_var=0.02, ignore_frac=0.2), 0.7,
     "mean", True, 10, 1024, True),
    (_w("f32_bias_bm", 100, 50, 777, "f32", bias_var=0.02, ignore_frac=0.1), 2.0, "batchmean",
     True, None, 0, False),
    (_w("f32_none", 257, 96, 2100, "f32"), 1.0, "none", False, 30, 512, False),
    # last vocabulary chunk 100 columns wide: with H <= 2048 the dlogits GEMM runs two
    # epilogue warps per lane quarter, and those of the second column half get no columns
    (_w("narrow_last_chunk_bias", 700, 192, 868, bias_var=0.02, ignore_frac=0.1), 1.3,
     "batchmean", True, None, 256, True),
    (_w("f16_narrow_last_chunk", 300, 128, 868, "f16", bias_var=0.02), 0.8, "sum", False,
     None, 256, False),
    # H > 2048: 4 epilogue warps, lane quarters 0 and 1 relayed through shared memory to
    # warps of the other two schedulers; ragged N, H and V (the last tile's relayed chunks
    # past V are skipped) and a 100-column last chunk
    (_w("h2312_relay_skip_bias", 300, 2312, 1000, bias_var=0.02, ignore_frac=0.1), 1.0,
     "batchmean", True, None, 0, True),
    (_w("h2304_relay_f16_topk", 257, 2304, 868, "f16"), 0.8, "none", False, 10, 256, False),
    (_w("relay_n1_v513", 1, 2112, 513, bias_var=0.02), 1.0, "sum", False, None, 0, False),
]


def _grad_out(reduction, n):
    if reduction == "none":
        g = torch.Generator().manual_seed(11)
        return (torch.rand(n, generator=g, dtype=torch.float64) + 0.5).float()
    return 0.75


def _labels(x, with_labels):
    return x["targets"] if with_labels else None


def run_kl_gpu(xd, q, labels, w, temperature, reduction, grad_out, vocab_chunk=0,
               skip_ignored=False, backward=True):
    err = torch.zeros((), dtype=torch.int32, device="cuda")
    f = api.flce_kl_forward_tensors(xd["hidden"], xd["weight"], q, labels, xd["bias"],
                                    w.ignore_index, temperature, 1e-10, reduction,
                                    err_word=err, skip_ignored=skip_ignored)
    out = {k: (None if t is None else t.detach().cpu()) for k, t in f.items()}
    if backward:
        go = (grad_out.cuda() if torch.is_tensor(grad_out)
              else torch.tensor(float(grad_out), dtype=torch.float32, device="cuda"))
        gh, gw, gb = api.flce_kl_backward_tensors(
            xd["hidden"], xd["weight"], q, f["lse_rows"], f["qsum_rows"], f["n_counted"], go,
            labels, xd["bias"], w.ignore_index, temperature, 1e-10, reduction, err_word=err,
            vocab_chunk=vocab_chunk, skip_ignored=skip_ignored)
        out["grad_hidden"], out["grad_weight"] = gh.cpu(), gw.cpu()
        out["grad_bias"] = None if gb is None else gb.cpu()
    torch.cuda.synchronize()
    out["err_word"] = int(err.item())
    return out


def _check_kl_scalar(out, ref, w, reduction, floor):
    """The reduced KL loss: rel 2e-3 / 1e-5 of itself plus the counted rows'
    floors and the fp32 rounding of its sum, divided as the reduction divides."""
    c = ref["counted"]
    nc = max(ref["n_counted"], 1)
    div = {"sum": 1.0, "batchmean": nc, "mean": nc * w.v}[reduction]
    assert_scalar_close("loss", float(out["loss"]), float(ref["loss_out"]),
                        TOL[w.dtype]["loss_rel"], float(floor[c].sum()) / div,
                        float(ref["loss"][c].abs().sum()) / div, nc)


@pytest.mark.parametrize("case", CASES, ids=[c[0].name for c in CASES])
def test_kl_parity(case):
    w, temp, reduction, with_labels, keep_top, chunk, skip = case
    x = make_inputs(w)
    q = make_teacher_probs(w, keep_top=keep_top)
    labels = _labels(x, with_labels)
    go = _grad_out(reduction, w.n)
    xd = to_dev(x)
    out = run_kl_gpu(xd, q.cuda(), None if labels is None else labels.cuda(), w, temp,
                     reduction, go, vocab_chunk=chunk, skip_ignored=skip)
    assert out["err_word"] == 0
    tol = TOL[w.dtype]
    ref = kl_oracle.forward(x["hidden"], x["weight"], q, x["bias"], labels, w.ignore_index,
                            temp, 1e-10, reduction)
    counted = ref["counted"]
    assert int(out["n_counted"]) == ref["n_counted"]
    floor = row_floor(w.h, kl_row_ops(ref))
    assert_rows_close("loss_rows", out["loss_rows"], ref["loss"], tol["loss_rel"], floor=floor)
    assert torch.all(out["loss_rows"][~counted] == 0)
    stat = counted if (skip and labels is not None) else None
    assert_rows_close("lse_rows", out["lse_rows"], ref["lse"], tol["loss_rel"], stat, floor)
    assert_rows_close("qsum_rows", out["qsum_rows"], ref["qsum"], 1e-5, stat)
    if stat is not None:
        assert bool(torch.isnan(out["lse_rows"][~counted]).all())
        assert bool(torch.isnan(out["qsum_rows"][~counted]).all())
    if reduction != "none":
        _check_kl_scalar(out, ref, w, reduction, floor)
    gref = kl_oracle.backward(x["hidden"], x["weight"], q, x["bias"], labels, w.ignore_index,
                              temp, 1e-10, reduction, go.double() if torch.is_tensor(go) else go,
                              magnitudes=True)
    kap = grad_kappas(w)
    for k in ("grad_hidden", "grad_weight") + (("grad_bias",) if x["bias"] is not None else ()):
        assert_grad_close(k, out[k], gref[k], tol, gref[k + "_mag"], kap[k])
    if labels is not None:
        assert torch.all(out["grad_hidden"][~counted] == 0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_onehot_teacher_equals_cross_entropy(dtype):
    """With a one-hot teacher at the targets and T = 1, KL(onehot || p) is the
    cross-entropy -log p_t, and d/dz is p - onehot: the KL path reproduces the
    separately pinned cross-entropy path (batchmean = mean over counted rows).
    Loss rows agree to rounding of the log of 1 in the approximate logarithm;
    lse rows and the gradients are bitwise equal."""
    w = _w("onehot", 700, 264, 3333, dtype, bias_var=0.02, ignore_frac=0.1)
    x = make_inputs(w)
    t = x["targets"]
    q = torch.zeros(w.n, w.v, dtype=w.torch_dtype)
    keep = t != w.ignore_index
    q[keep, t[keep]] = 1.0
    xd = to_dev(x)
    kl = run_kl_gpu(xd, q.cuda(), xd["targets"], w, 1.0, "batchmean", 0.75)
    ce_f = api.flce_forward_tensors(xd["hidden"], xd["weight"], xd["targets"], xd["bias"],
                                    w.ignore_index, reduction="mean")
    go = torch.tensor(0.75, dtype=torch.float32, device="cuda")
    ce_g = api.flce_backward_tensors(xd["hidden"], xd["weight"], xd["targets"],
                                     ce_f["lse_rows"], ce_f["n_valid"], go, xd["bias"],
                                     w.ignore_index, reduction="mean")
    torch.cuda.synchronize()
    assert torch.equal(kl["lse_rows"], ce_f["lse_rows"].cpu())
    assert torch.allclose(kl["loss_rows"], ce_f["loss_rows"].cpu(), rtol=1e-6, atol=1e-6)
    assert abs(float(kl["loss"]) - float(ce_f["loss"])) <= 1e-6 * abs(float(ce_f["loss"]))
    assert torch.equal(kl["grad_hidden"], ce_g[0].cpu())
    assert torch.equal(kl["grad_weight"], ce_g[1].cpu())
    assert torch.equal(kl["grad_bias"], ce_g[2].cpu())


def test_kl_empty_and_all_ignored():
    w = _w("empty", 0, 64, 1000)
    x = make_inputs(w)
    xd = to_dev(x)
    q = torch.empty(0, w.v, dtype=torch.bfloat16, device="cuda")
    for reduction, expect in (("batchmean", math.nan), ("sum", 0.0), ("mean", math.nan)):
        out = run_kl_gpu(xd, q, xd["targets"], w, 1.0, reduction, 1.0)
        assert int(out["n_counted"]) == 0
        got = float(out["loss"])
        assert (math.isnan(got) if math.isnan(expect) else got == expect)
        assert torch.all(out["grad_weight"] == 0)
    w = _w("all_ignored", 300, 64, 1000, ignore_frac=1.0)
    x = make_inputs(w)
    xd = to_dev(x)
    q = make_teacher_probs(w).cuda()
    for skip in (False, True):
        out = run_kl_gpu(xd, q, xd["targets"], w, 1.0, "sum", 1.0, skip_ignored=skip)
        assert int(out["n_counted"]) == 0 and float(out["loss"]) == 0.0
        assert torch.all(out["loss_rows"] == 0)
        for k in ("grad_hidden", "grad_weight"):
            assert torch.all(out[k] == 0), k


def test_kl_autograd_matches_raw_calls_and_repeats_bitwise():
    w = _w("autograd", 600, 192, 5000, bias_var=0.02, ignore_frac=0.2)
    x = make_inputs(w)
    xd = to_dev(x)
    q = make_teacher_probs(w, keep_top=100).cuda()
    raw = run_kl_gpu(xd, q, xd["targets"], w, 1.3, "batchmean", 1.0, skip_ignored=True)
    again = run_kl_gpu(xd, q, xd["targets"], w, 1.3, "batchmean", 1.0, skip_ignored=True)
    for k in ("loss", "loss_rows", "grad_hidden", "grad_weight", "grad_bias"):
        assert torch.equal(raw[k], again[k]), k
    h = xd["hidden"].clone().requires_grad_(True)
    wt = xd["weight"].clone().requires_grad_(True)
    b = xd["bias"].clone().requires_grad_(True)
    loss = fused_linear_kl_div(h, wt, q, xd["targets"], b, temperature=1.3)
    loss.backward()
    assert torch.equal(loss.detach().cpu(), raw["loss"])
    assert torch.equal(h.grad.cpu(), raw["grad_hidden"])
    assert torch.equal(wt.grad.cpu(), raw["grad_weight"])
    assert torch.equal(b.grad.cpu(), raw["grad_bias"])
    # vocab_chunk reaches the backward: 1024 gives five chunks, bitwise the raw calls
    raw_c = run_kl_gpu(xd, q, xd["targets"], w, 1.3, "batchmean", 1.0, vocab_chunk=1024,
                       skip_ignored=True)
    for t in (h, wt, b):
        t.grad = None
    loss = fused_linear_kl_div(h, wt, q, xd["targets"], b, temperature=1.3, vocab_chunk=1024)
    loss.backward()
    assert torch.equal(h.grad.cpu(), raw_c["grad_hidden"])
    assert torch.equal(wt.grad.cpu(), raw_c["grad_weight"])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_kl_degenerate_shapes_and_teachers(dtype):
    """V = 1: p = 1, so loss_i = q_i log max(q_i, eps) and D = g (Q - q) / T = 0
    exactly. N = 1. A teacher row of zeros contributes 0 and no gradient.
    Temperatures 0.05 (sharp) and 20 (flat). Each case against the oracle,
    V = 1 and the zero row also against their closed forms.

    At T = 0.05 with bf16 inputs |D| reaches ~13 and grad_hidden = D @ W
    cancels in some entries, so rounding D to bf16 moves such an entry by up
    to 2^-8 sum_j |D_j||W_jk| whatever the kernel does: the elementwise bar's
    kappa * M term (tests/_parity.py) bounds exactly that."""
    tol = TOL[dtype]
    # V = 1
    w = _w("v1", 40, 16, 1, dtype)
    x = make_inputs(w)
    q = torch.rand(w.n, 1, generator=torch.Generator().manual_seed(3)).to(w.torch_dtype)
    out = run_kl_gpu(to_dev(x), q.cuda(), None, w, 1.0, "sum", 1.0)
    qd = q.double().reshape(-1)
    expect = (qd * torch.log(qd.clamp_min(1e-10))).sum()
    # fp32 terms q log q (|.| <= 1/e) summed over the rows
    terms = (qd * torch.log(qd.clamp_min(1e-10))).abs()
    assert_scalar_close("loss", float(out["loss"]), float(expect), tol["loss_rel"],
                        float(row_floor(w.h, terms).sum()), float(terms.sum()), w.n)
    for k in ("grad_hidden", "grad_weight"):
        assert torch.all(out[k] == 0), k
    # N = 1 and the temperatures
    for temp in (0.05, 20.0):
        w = _w("n1", 1, 64, 777, dtype, bias_var=0.02)
        x = make_inputs(w)
        q = make_teacher_probs(w, keep_top=5)
        out = run_kl_gpu(to_dev(x), q.cuda(), None, w, temp, "batchmean", 1.0)
        ref = kl_oracle.forward(x["hidden"], x["weight"], q, x["bias"], None, -100, temp, 1e-10,
                                "batchmean")
        assert_rows_close("loss_rows", out["loss_rows"], ref["loss"], tol["loss_rel"],
                          floor=row_floor(w.h, kl_row_ops(ref)))
        gref = kl_oracle.backward(x["hidden"], x["weight"], q, x["bias"], None, -100, temp,
                                  1e-10, "batchmean", 1.0, magnitudes=True)
        kap = grad_kappas(w)
        for k in ("grad_hidden", "grad_weight", "grad_bias"):
            assert_grad_close(k, out[k], gref[k], tol, gref[k + "_mag"], kap[k])
    # a zero teacher row among ordinary ones
    w = _w("zero_row", 130, 64, 1000, dtype)
    x = make_inputs(w)
    q = make_teacher_probs(w)
    q[7] = 0
    out = run_kl_gpu(to_dev(x), q.cuda(), None, w, 1.0, "none", torch.ones(w.n))
    assert float(out["loss_rows"][7]) == 0.0 and float(out["qsum_rows"][7]) == 0.0
    assert torch.all(out["grad_hidden"][7] == 0)
    ref = kl_oracle.forward(x["hidden"], x["weight"], q, None, None, -100, 1.0, 1e-10, "none")
    assert_rows_close("loss_rows", out["loss_rows"], ref["loss"], tol["loss_rel"],
                      floor=row_floor(w.h, kl_row_ops(ref)))


def test_kl_grad_weight_fp32_output():
    """grad_weight kept in fp32 (grad_weight_dtype=float32) for the KL
    divergence: same bars as bf16 (D is still bf16), and it equals the bf16
    output up to that output's rounding."""
    w = _w("gw32", 300, 136, 1000, bias_var=0.02, ignore_frac=0.1)
    x = make_inputs(w)
    q = make_teacher_probs(w)
    xd = to_dev(x)
    qd, lab = q.cuda(), xd["targets"]
    f = api.flce_kl_forward_tensors(xd["hidden"], xd["weight"], qd, lab, xd["bias"],
                                    temperature=1.3)
    go = torch.tensor(1.0, dtype=torch.float32, device="cuda")
    outs = {}
    for dt in (None, torch.float32):
        outs[dt] = api.flce_kl_backward_tensors(xd["hidden"], xd["weight"], qd, f["lse_rows"],
                                                f["qsum_rows"], f["n_counted"], go, lab,
                                                xd["bias"], temperature=1.3,
                                                grad_weight_dtype=dt)
    torch.cuda.synchronize()
    gw32 = outs[torch.float32][1]
    assert gw32.dtype == torch.float32
    assert torch.equal(gw32.to(torch.bfloat16), outs[None][1])
    gref = kl_oracle.backward(x["hidden"], x["weight"], q, x["bias"], x["targets"], -100, 1.3,
                              1e-10, "batchmean", 1.0, magnitudes=True)
    assert_grad_close("grad_weight fp32", gw32.cpu(), gref["grad_weight"], TOL["bf16"],
                      gref["grad_weight_mag"], grad_kappas(w)["grad_weight"])
