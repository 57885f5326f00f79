"""The oracle reproduces its stored tiny fixtures, and the pure-Python brute
force agrees with them independently (forward quantities)."""
import json
import os

import pytest
import torch

import oracle
from oracle import brute

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
with open(os.path.join(HERE, "tiny_oracle.json")) as fh:
    FIX = json.load(fh)["cases"]


def _t(x):
    return None if x is None else torch.tensor(x, dtype=torch.float64)


@pytest.mark.parametrize("c", FIX, ids=[c["name"] for c in FIX])
def test_oracle_reproduces_fixture(c):
    h, w, b = _t(c["hidden"]), _t(c["weight"]), _t(c["bias"])
    t = torch.tensor(c["targets"], dtype=torch.int64)
    args = (h, w, t, b, -100, c["logit_scale"], c["softcap"], c["reduction"])
    f = oracle.forward(*args)
    g = oracle.backward(*args, 1.0)
    assert torch.allclose(f["loss"], _t(c["loss_rows"]), rtol=1e-12, atol=1e-15)
    assert torch.allclose(f["lse"], _t(c["lse"]), rtol=1e-12)
    assert f["argmax"].tolist() == c["argmax"]
    assert f["loss_out"] == pytest.approx(c["loss_out"], rel=1e-12)
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        if c[k] is not None:
            assert torch.allclose(g[k], _t(c[k]), rtol=1e-11, atol=1e-16)


@pytest.mark.parametrize("c", FIX, ids=[c["name"] for c in FIX])
def test_brute_force_agrees_with_fixture(c):
    rows = brute.per_row(c["hidden"], c["weight"], c["targets"], c["bias"], -100,
                         c["logit_scale"], c["softcap"])
    for r, l, e, a in zip(rows, c["loss_rows"], c["entropy"], c["argmax"]):
        assert r["loss"] == pytest.approx(l, rel=1e-12, abs=1e-15)
        assert r["entropy"] == pytest.approx(e, rel=1e-12)
        assert r["argmax"] == a
    acc, ent = brute.metrics(c["hidden"], c["weight"], c["targets"], c["bias"], -100,
                             c["logit_scale"], c["softcap"])
    assert acc == pytest.approx(c["mean_token_accuracy"])
    assert ent == pytest.approx(c["entropy_mean"], rel=1e-12)


with open(os.path.join(HERE, "tiny_kl_oracle.json")) as fh:
    KL_FIX = json.load(fh)["cases"]


@pytest.mark.parametrize("c", KL_FIX, ids=[c["name"] for c in KL_FIX])
def test_kl_oracle_reproduces_fixture(c):
    from oracle import kl_oracle

    h, w, b, q = _t(c["hidden"]), _t(c["weight"]), _t(c["bias"]), _t(c["target_probs"])
    lab = None if c["labels"] is None else torch.tensor(c["labels"], dtype=torch.int64)
    args = (h, w, q, b, lab, -100, c["temperature"], 1e-10, c["reduction"])
    f = kl_oracle.forward(*args)
    g = kl_oracle.backward(*args, 1.0)
    assert torch.allclose(f["loss"], _t(c["loss_rows"]), rtol=1e-12, atol=1e-15)
    assert torch.allclose(f["lse"], _t(c["lse"]), rtol=1e-12)
    assert torch.allclose(f["qsum"], _t(c["qsum"]), rtol=1e-12)
    assert f["n_counted"] == c["n_counted"]
    assert f["loss_out"] == pytest.approx(c["loss_out"], rel=1e-12)
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        if c[k] is not None:
            assert torch.allclose(g[k], _t(c[k]), rtol=1e-11, atol=1e-16)


@pytest.mark.parametrize("c", KL_FIX, ids=[c["name"] for c in KL_FIX])
def test_kl_brute_force_agrees_with_fixture(c):
    rows = brute.kl_per_row(c["hidden"], c["weight"], c["target_probs"], c["bias"], c["labels"],
                            -100, c["temperature"], 1e-10)
    for r, l in zip(rows, c["loss_rows"]):
        assert r == pytest.approx(l, rel=1e-11, abs=1e-14)
