"""Pins of the oracles' gradient magnitudes (``backward(..., magnitudes=True)``):
for each gradient entry, the sum of the absolute values of the terms it adds
up (sum_j |D_ij||W_jk|, sum_i |D_ij||h_ik|, sum_i |D_ij|). The GPU parity
tests bound an entry's error by a multiple of it, so a mistake here would
loosen or tighten every gradient bar.

Pinned against what does not depend on how the oracle forms them:
  * the triangle inequality: |grad| <= magnitude, entry by entry;
  * sign-coherent entries: where every term has the same sign the magnitude
    is |grad| exactly (non-negative hidden and a vocabulary row that is no
    row's target: every D_ij = g_i p_ij dz/dlin >= 0);
  * a closed form for the gap: with non-negative weight (or hidden) and no
    softcap, the only negative term of row i is its target's,
    D_{i,t_i} = g_i (p_{i,t_i} - 1) s, so magnitude - grad = 2 g_i (1 - p_{i,t_i}) s
    times the target's weight row (or the row's hidden values), with
    p_{i,t_i} from the brute force's explicit softmax;
and a planted mistake in each place an absolute value is taken must fail
one of them.
"""
import pytest
import torch

import oracle
from oracle import brute, flce_oracle, kl_oracle

F64 = torch.float64


def _inputs(n, h, v, seed, bias=True, ignore=(1,)):
    g = torch.Generator().manual_seed(seed)
    hid = torch.randn(n, h, generator=g, dtype=F64)
    w = torch.randn(v, h, generator=g, dtype=F64) * 0.6
    b = torch.randn(v, generator=g, dtype=F64) * 0.3 if bias else None
    t = torch.randint(0, v // 2, (n,), generator=g)  # the upper half is no row's target
    for i in ignore:
        t[i] = -100
    return hid, w, b, t


@pytest.mark.parametrize("softcap,eps,lam,red", [(None, 0.0, 0.0, "mean"), (3.0, 0.1, 1e-2, "sum"),
                                                 (2.0, 0.0, 0.0, "none")])
def test_triangle_inequality(softcap, eps, lam, red):
    hid, w, b, t = _inputs(9, 6, 13, 1)
    go = torch.linspace(0.5, 1.5, 9, dtype=F64) if red == "none" else 0.8
    g = oracle.backward(hid, w, t, b, -100, 0.7, softcap, red, go, magnitudes=True,
                        label_smoothing=eps, z_loss=lam)
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        assert bool((g[k].abs() <= g[k + "_mag"] * (1 + 1e-12) + 1e-300).all()), k
        assert bool((g[k + "_mag"] > 0).any()), k


def test_sign_coherent_entries_equal_the_gradient():
    hid, w, b, t = _inputs(8, 5, 12, 2)
    hid = hid.abs()
    g = oracle.backward(hid, w, t, b, -100, 0.9, 2.5, "sum", 1.0, magnitudes=True)
    cols = torch.arange(6, 12)  # no row targets these vocabulary rows
    assert torch.allclose(g["grad_weight_mag"][cols], g["grad_weight"][cols], rtol=1e-12, atol=0)
    assert torch.allclose(g["grad_bias_mag"][cols], g["grad_bias"][cols], rtol=1e-12, atol=0)


def _target_gap(hid, w, b, t, scale, red):
    """2 g_i (1 - p_{i,t_i}) s per valid row, p from the brute force."""
    rows = brute.per_row(hid.tolist(), w.tolist(), t.tolist(), b.tolist(), -100, scale, None)
    valid = t != -100
    nv = int(valid.sum())
    g = 1.0 / nv if red == "mean" else 1.0
    gap = torch.zeros(t.numel(), dtype=F64)
    for i, r in enumerate(rows):
        if r["valid"]:
            gap[i] = 2.0 * g * (1.0 - r["p"][int(t[i])]) * scale
    return gap, valid


@pytest.mark.parametrize("red", ["mean", "sum"])
def test_closed_form_gap(red):
    hid, w, b, t = _inputs(7, 4, 10, 3)
    scale = 0.8
    gap, valid = _target_gap(hid, w, b, t, scale, red)
    # grad_hidden with a non-negative weight
    wp = w.abs()
    g = oracle.backward(hid, wp, t, b, -100, scale, None, red, 1.0, magnitudes=True)
    gap_p, _ = _target_gap(hid, wp, b, t, scale, red)
    expect = torch.zeros_like(g["grad_hidden"])
    expect[valid] = gap_p[valid, None] * wp[t[valid]]
    assert torch.allclose(g["grad_hidden_mag"] - g["grad_hidden"], expect, rtol=1e-10, atol=1e-14)
    # grad_weight and grad_bias with a non-negative hidden
    hp = hid.abs()
    g = oracle.backward(hp, w, t, b, -100, scale, None, red, 1.0, magnitudes=True)
    gap_h, _ = _target_gap(hp, w, b, t, scale, red)
    expect_w = torch.zeros_like(g["grad_weight"])
    expect_b = torch.zeros_like(g["grad_bias"])
    for i in torch.nonzero(valid).flatten().tolist():
        expect_w[t[i]] += gap_h[i] * hp[i]
        expect_b[t[i]] += gap_h[i]
    assert torch.allclose(g["grad_weight_mag"] - g["grad_weight"], expect_w, rtol=1e-10,
                          atol=1e-14)
    assert torch.allclose(g["grad_bias_mag"] - g["grad_bias"], expect_b, rtol=1e-10, atol=1e-14)


def test_kl_triangle_and_onehot_gap():
    """KL: the triangle inequality on a dense teacher; with a one-hot teacher
    at the targets D = g (p - onehot) / T, so the gap is the cross-entropy's
    with s = 1/T and p_t = exp(-loss_i) from the brute force's KL rows."""
    hid, w, b, t = _inputs(6, 5, 11, 4, ignore=())
    q = torch.softmax(torch.randn(6, 11, generator=torch.Generator().manual_seed(9),
                                  dtype=F64), dim=1)
    g = kl_oracle.backward(hid, w, q, b, None, -100, 1.3, 1e-10, "sum", 1.0, magnitudes=True)
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        assert bool((g[k].abs() <= g[k + "_mag"] * (1 + 1e-12)).all()), k
    temp = 1.7
    onehot = torch.zeros(6, 11, dtype=F64)
    onehot[torch.arange(6), t] = 1.0
    wp = w.abs()
    g = kl_oracle.backward(hid, wp, onehot, b, None, -100, temp, 1e-10, "sum", 1.0,
                           magnitudes=True)
    rows = brute.kl_per_row(hid.tolist(), wp.tolist(), onehot.tolist(), b.tolist(), None, -100,
                            temp)
    p_t = torch.exp(-torch.tensor(rows, dtype=F64))
    expect = 2.0 * (1.0 - p_t)[:, None] / temp * wp[t]
    assert torch.allclose(g["grad_hidden_mag"] - g["grad_hidden"], expect, rtol=1e-10, atol=1e-14)


def _mut_no_abs_left(a, b):
    return a @ b.abs()


def _mut_no_abs_right(a, b):
    return a.abs() @ b


def _mut_abs_of_sum(a, b):
    return (a @ b).abs()


@pytest.mark.parametrize("mutant", [_mut_no_abs_left, _mut_no_abs_right, _mut_abs_of_sum],
                         ids=lambda m: m.__name__)
@pytest.mark.parametrize("module", [flce_oracle, kl_oracle], ids=["ce", "kl"])
def test_planted_mistakes(monkeypatch, module, mutant):
    def pins():
        try:
            for args in ((None, 0.0, 0.0, "mean"), (3.0, 0.1, 1e-2, "sum")):
                test_triangle_inequality(*args)
            test_sign_coherent_entries_equal_the_gradient()
            for red in ("mean", "sum"):
                test_closed_form_gap(red)
            test_kl_triangle_and_onehot_gap()
        except AssertionError:
            return False
        return True

    assert pins()
    monkeypatch.setattr(module, "_abs_terms", mutant)
    assert not pins(), f"{module.__name__}: {mutant.__name__} went unnoticed"
