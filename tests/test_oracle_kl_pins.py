"""Pins of the fused linear KL divergence oracle (Liger-Kernel pull request
#1423, FusedLinearKLDivLoss: KL(Q || P) against explicit teacher
probabilities, with temperature, eps clamp, batchmean/mean/sum and ignored
rows): a pure-Python brute force, central finite differences of it,
torch.nn.functional.kl_div with autograd, closed forms, and planted
mistakes that the pins must catch."""
import math

import pytest
import torch

from oracle import brute, kl_oracle

# torch announces that its kl_div 'mean' will change meaning; these pins compare
# against today's definition (the total over all N x V entries divided by N x V)
pytestmark = pytest.mark.filterwarnings("ignore:reduction. 'mean' divides:UserWarning")

F64 = torch.float64


def _inputs(n, h, v, bias=True, seed=0, ignore=0.25, sharp=1.0):
    g = torch.Generator().manual_seed(seed)
    hid = torch.randn(n, h, generator=g, dtype=F64)
    w = torch.randn(v, h, generator=g, dtype=F64) / math.sqrt(h)
    b = torch.randn(v, generator=g, dtype=F64) * 0.3 if bias else None
    q = torch.softmax(sharp * torch.randn(n, v, generator=g, dtype=F64), dim=1)
    # rows that do not sum to 1 (as bf16 teacher rows do not exactly), so that a
    # dropped sum_j q_ij factor is visible; the definition holds for any q >= 0
    q = q * (0.5 + torch.rand(n, 1, generator=g, dtype=F64))
    labels = torch.zeros(n, dtype=torch.int64)
    labels[torch.randperm(n, generator=g)[:int(round(ignore * n))]] = -100
    return hid, w, b, q, labels


CASES = [("batchmean", 1.0), ("sum", 2.0), ("mean", 0.5), ("none", 1.5)]


@pytest.mark.parametrize("reduction,temp", CASES)
def test_brute_force_forward(reduction, temp):
    hid, w, b, q, lab = _inputs(9, 6, 13)
    f = kl_oracle.forward(hid, w, q, b, lab, -100, temp, 1e-10, reduction)
    rows = brute.kl_per_row(hid.tolist(), w.tolist(), q.tolist(), b.tolist(), lab.tolist(),
                            -100, temp)
    for i, r in enumerate(rows):
        assert f["loss"][i].item() == pytest.approx(r, rel=1e-12, abs=1e-15)


def _fd(reduction, temp, mod=kl_oracle, n_probe=5, step=1e-5):
    hid, w, b, q, lab = _inputs(8, 5, 11, seed=2)
    g = torch.Generator().manual_seed(9)
    row_g = torch.rand(8, generator=g, dtype=F64) + 0.5 if reduction == "none" else None
    go = row_g if row_g is not None else 0.8
    grads = mod.backward(hid, w, q, b, lab, -100, temp, 1e-10, reduction, go)
    scale = 1.0 if row_g is not None else 0.8

    def L(hh, ww, bb):
        return scale * brute.kl_loss(hh.tolist(), ww.tolist(), q.tolist(), bb.tolist(),
                                     lab.tolist(), -100, temp, 1e-10, reduction,
                                     None if row_g is None else row_g.tolist())

    worst = 0.0
    for name, key, base in (("h", "grad_hidden", hid), ("w", "grad_weight", w), ("b", "grad_bias", b)):
        for _ in range(n_probe):
            k = int(torch.randint(0, base.numel(), (1,), generator=g))
            plus, minus = base.clone().reshape(-1), base.clone().reshape(-1)
            plus[k] += step
            minus[k] -= step
            args = {"h": hid, "w": w, "b": b}
            args[name] = plus.reshape(base.shape)
            lp = L(args["h"], args["w"], args["b"])
            args[name] = minus.reshape(base.shape)
            lm = L(args["h"], args["w"], args["b"])
            fd = (lp - lm) / (2 * step)
            an = grads[key].reshape(-1)[k].item()
            worst = max(worst, abs(fd - an) / max(1e-6, abs(fd), abs(an)))
    return worst


@pytest.mark.parametrize("reduction,temp", CASES)
def test_finite_differences(reduction, temp):
    assert _fd(reduction, temp) < 1e-6


@pytest.mark.parametrize("reduction", ["batchmean", "sum", "mean"])
def test_torch_kl_div(reduction):
    """torch.nn.functional.kl_div(log_softmax(x / T), q) with autograd, every
    row counted (torch's batchmean and mean count all rows)."""
    temp = 1.7
    hid, w, b, q, _ = _inputs(12, 7, 19, seed=4)
    hr, wr, br = (t.clone().requires_grad_(True) for t in (hid, w, b))
    logp = torch.log_softmax(torch.nn.functional.linear(hr, wr, br) / temp, dim=1)
    ref = torch.nn.functional.kl_div(logp, q, reduction=reduction)
    ref.backward()
    f = kl_oracle.forward(hid, w, q, b, None, -100, temp, 1e-30, reduction)
    assert f["loss_out"] == pytest.approx(ref.item(), rel=1e-12)
    gr = kl_oracle.backward(hid, w, q, b, None, -100, temp, 1e-30, reduction, 1.0)
    assert torch.allclose(gr["grad_hidden"], hr.grad, rtol=1e-11, atol=1e-15)
    assert torch.allclose(gr["grad_weight"], wr.grad, rtol=1e-11, atol=1e-15)
    assert torch.allclose(gr["grad_bias"], br.grad, rtol=1e-11, atol=1e-15)


def test_teacher_equals_student():
    """Q = P: the divergence is 0 and so is every gradient."""
    hid, w, b, _, lab = _inputs(10, 6, 17, seed=5)
    temp = 1.3
    q = torch.softmax((hid @ w.T + b) / temp, dim=1)
    f = kl_oracle.forward(hid, w, q, b, lab, -100, temp, 1e-30, "sum")
    assert abs(f["loss_out"]) < 1e-13
    gr = kl_oracle.backward(hid, w, q, b, lab, -100, temp, 1e-30, "sum", 1.0)
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        assert float(gr[k].abs().max()) < 1e-14


def test_zero_weight_closed_form():
    """W = 0, b = 0: P is uniform, so loss_i = sum_j q_ij log q_ij +
    log V * sum_j q_ij; a zero probability adds 0."""
    n, h, v = 6, 4, 9
    hid, _, _, q, _ = _inputs(n, h, v, bias=False, seed=6)
    q[0] = 0.0
    q[0, 3] = 1.0
    f = kl_oracle.forward(hid, torch.zeros(v, h, dtype=F64), q, None, None, -100, 1.0, 1e-10,
                          "none")
    for i in range(n):
        expect = (sum(float(x) * math.log(float(x)) for x in q[i] if x > 0)
                  + math.log(v) * float(q[i].sum()))
        assert f["loss"][i].item() == pytest.approx(expect, rel=1e-12, abs=1e-14)


def _mut_no_qsum(hidden, weight, target_probs, bias=None, labels=None, ignore_index=-100,
                 temperature=1.0, eps=1e-10, reduction="batchmean", grad_out=1.0, rows=None,
                 vocab_rows=None):
    # D = g (p - q) / T instead of g (p * sum(q) - q) / T
    n, v = hidden.shape[0], weight.shape[0]
    g = kl_oracle.row_weights(labels, n, v, ignore_index, reduction, grad_out)
    z = (hidden @ weight.T + (0 if bias is None else bias)) / temperature
    p = torch.softmax(z, dim=1)
    d = (p - target_probs) * (g / temperature)[:, None]
    return {"grad_hidden": d @ weight, "grad_weight": d.T @ hidden,
            "grad_bias": None if bias is None else d.sum(dim=0)}


def _mut_temperature(hidden, weight, target_probs, bias=None, labels=None, ignore_index=-100,
                     temperature=1.0, eps=1e-10, reduction="batchmean", grad_out=1.0, rows=None,
                     vocab_rows=None):
    r = ORIG_BACKWARD(hidden, weight, target_probs, bias, labels, ignore_index, temperature, eps,
                      reduction, grad_out, rows, vocab_rows)
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        if r[k] is not None:
            r[k] = r[k] * temperature  # drops the 1/T factor
    return r


ORIG_BACKWARD = kl_oracle.backward


@pytest.mark.parametrize("mutant", [_mut_no_qsum, _mut_temperature])
def test_planted_mistakes(monkeypatch, mutant):
    monkeypatch.setattr(kl_oracle, "backward", mutant)
    worst = max(_fd(red, t, mod=kl_oracle, n_probe=3) for red, t in CASES)
    assert worst > 1e-6, f"{mutant.__name__} went unnoticed"


ORIG_FORWARD = kl_oracle.forward


def _mut_fwd_no_clamp(hidden, weight, target_probs, bias=None, labels=None, ignore_index=-100,
                      temperature=1.0, eps=1e-10, reduction="batchmean", rows=None):
    # log q without the eps clamp: a zero probability gives 0 * log 0 = NaN
    return ORIG_FORWARD(hidden, weight, target_probs, bias, labels, ignore_index, temperature,
                        0.0, reduction, rows)


def _mut_fwd_mean_as_batchmean(hidden, weight, target_probs, bias=None, labels=None,
                               ignore_index=-100, temperature=1.0, eps=1e-10,
                               reduction="batchmean", rows=None):
    red = "batchmean" if reduction == "mean" else reduction
    return ORIG_FORWARD(hidden, weight, target_probs, bias, labels, ignore_index, temperature,
                        eps, red, rows)


def _mut_fwd_no_lse(hidden, weight, target_probs, bias=None, labels=None, ignore_index=-100,
                    temperature=1.0, eps=1e-10, reduction="batchmean", rows=None):
    # sum q (log q - z): the lse * sum q term dropped
    r = ORIG_FORWARD(hidden, weight, target_probs, bias, labels, ignore_index, temperature, eps,
                     reduction, rows)
    keep = r["counted"].to(F64)
    r["loss"] = r["loss"] - r["lse"] * r["qsum"] * keep
    if rows is None and reduction != "none":
        scale = r["loss_out"] / float(ORIG_FORWARD(hidden, weight, target_probs, bias, labels,
                                                   ignore_index, temperature, eps, "sum")
                                      ["loss_out"])
        r["loss_out"] = float(r["loss"].sum()) * scale
    return r


def _forward_pins():
    for red, t in CASES:
        test_brute_force_forward(red, t)
    test_zero_weight_closed_form()
    for red in ("batchmean", "sum", "mean"):
        test_torch_kl_div(red)


@pytest.mark.parametrize("mutant", [_mut_fwd_no_clamp, _mut_fwd_mean_as_batchmean,
                                    _mut_fwd_no_lse])
def test_planted_forward_mistakes(monkeypatch, mutant):
    monkeypatch.setattr(kl_oracle, "forward", mutant)
    with pytest.raises(AssertionError):
        _forward_pins()
