"""Full-size parity at the three large workloads, in the launch configuration
bench.py times (default vocabulary chunking, one stream, ignored rows left
out of the contractions).

The oracle runs its fp64 forward over every row: per-row loss, lse, entropy
and argmax are compared for all N rows, and the reduced loss and metrics
exactly. The gradients are compared on samples the oracle computes one by
one:
  * 512 grad_hidden rows, stratified: first and last rows, ignored rows,
    rows whose target is a peaked (x8) weight row, the rest random;
  * 256 grad_weight (and grad_bias) rows: vocabulary ids 0, 1, V-1, tile
    and chunk boundaries, peaked rows, targets of sampled rows, the rest
    random.
Plus a property that holds at any size: with softcap off and logit_scale 1,
sum_j grad_weight[j, :] = 0 up to bf16 rounding. The fused linear KL
divergence gets the same treatment at the Llama-3 head shape.

These take minutes of host fp64 work each (the oracle's full forward is
2·N·H·V multiply-adds).
"""
import pytest
import torch

import oracle
from _parity import TOL, check_backward, check_forward, grad_kappas, oracle_args, run_gpu, to_dev
from linear_cross_entropy_vocab_gb300.workloads import WORKLOADS, Workload, make_inputs, peaked_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]



def default_chunk(n, v, elem=2, budget=512 << 20):
    """The library's default backward chunk width (include/flce.h, vocab_chunk):
    at least five equal chunks of whole 256-column tiles (one per tile below
    five tiles), more while a chunk's n x width buffer exceeds 512 MiB. Used
    only to place sampled vocabulary rows at chunk boundaries."""
    v_round = -(-v // 256) * 256
    nch = max(-(-(max(n, 1) * elem * v_round) // budget), min(5, v_round // 256))
    width = -(-(-(-v // nch)) // 256) * 256
    while width > 256 and width * max(n, 1) * elem > budget:
        nch += 1
        width = -(-(-(-v // nch)) // 256) * 256
    return min(width, v_round)


def _sample_rows(w, targets, peaked, k=512, seed=11):
    n = w.n
    g = torch.Generator().manual_seed(seed)
    picks = [0, 1, n - 1, n - 2, min(n - 1, 127), min(n - 1, 128)]
    picks += torch.nonzero(targets == w.ignore_index).flatten()[:48].tolist()
    if peaked.numel():
        hit = torch.isin(targets, peaked)
        picks += torch.nonzero(hit).flatten()[:64].tolist()
    picks += torch.randperm(n, generator=g)[:k].tolist()
    out = []
    for r in picks:
        if r not in out:
            out.append(int(r))
    return sorted(out[:k])


def _sample_vocab(w, targets, rows, peaked, k=256, seed=12):
    v = w.v
    g = torch.Generator().manual_seed(seed)
    chunk = default_chunk(w.n, v)
    picks = [0, 1, v - 1, v - 2, 255, 256, 257]
    c = chunk
    while c < v:
        picks += [c - 1, c]
        c += chunk
    picks += peaked[:32].tolist()
    t = targets[rows]
    picks += t[(t >= 0) & (t < v)][:48].tolist()
    picks += torch.randperm(v, generator=g)[:k].tolist()
    out = []
    for j in picks:
        if 0 <= j < v and j not in out:
            out.append(int(j))
    return sorted(out[:k])


@pytest.mark.parametrize("name", ["llama3_head_bf16", "softcap_bf16", "long_bf16"])
def test_fullsize_parity(name):
    w = WORKLOADS[name]
    x = make_inputs(w)
    xd = to_dev(x)
    tol = TOL[w.dtype]
    if name == "long_bf16":
        # first phase of this workload: forward only, reduction none
        w_none = w.with_shape(reduction="none")
        fwd_none = run_gpu(xd, w_none, backward=False, skip_ignored=True)
    out = run_gpu(xd, w, grad_out=1.0, skip_ignored=True)
    assert out["err_word"] == 0
    ref = oracle.forward(*oracle_args(x, w))
    check_forward(out, ref, w, tol, skipped=True)
    if name == "long_bf16":
        keep = x["targets"] != w.ignore_index
        assert torch.equal(fwd_none["loss_rows"], out["loss_rows"])
        assert torch.equal(fwd_none["lse_rows"][keep], out["lse_rows"][keep])
    peaked = peaked_rows(w)
    rows = _sample_rows(w, x["targets"], peaked)
    vocab = _sample_vocab(w, x["targets"], rows, peaked)
    gref = oracle.backward(*oracle_args(x, w), 1.0, lse=ref["lse"], rows=rows, vocab_rows=vocab,
                           magnitudes=True)
    sampled = {
        "grad_hidden": out["grad_hidden"][rows],
        "grad_weight": out["grad_weight"][vocab],
        "grad_bias": None if out["grad_bias"] is None else out["grad_bias"][vocab],
    }
    check_backward(sampled, gref, tol, x["bias"] is not None, grad_kappas(w))
    if w.softcap is None and w.logit_scale == 1.0:
        gw = out["grad_weight"].double()
        col = gw.sum(dim=0).abs()
        mag = gw.abs().sum(dim=0)
        assert bool((col <= 1e-2 * mag + 1e-12).all()), float((col / mag).max())


def test_fullsize_kl_parity():
    """The fused linear KL divergence at the Llama-3 head shape, in the
    configuration `bench.py --kl` times: teacher probabilities from
    make_teacher_probs, the workload's targets as labels (2 % ignored, left
    out of the contractions), T = 1, batchmean. Per-row loss, lse and sum q
    for all N rows; gradients on sampled rows; and, at any size,
    sum_j grad_weight[j, :] = 0 (each counted row's p * sum q - q sums to 0
    over the vocabulary)."""
    from _parity import (assert_grad_close, assert_rows_close, assert_scalar_close, kl_row_ops,
                         row_floor)
    from linear_cross_entropy_vocab_gb300 import api
    from linear_cross_entropy_vocab_gb300.workloads import make_teacher_probs
    from oracle import kl_oracle

    w = WORKLOADS["llama3_head_bf16"]
    x = make_inputs(w)
    q = make_teacher_probs(w)
    xd = to_dev(x)
    qd = q.cuda()
    tol = TOL[w.dtype]
    err = torch.zeros((), dtype=torch.int32, device="cuda")
    f = api.flce_kl_forward_tensors(xd["hidden"], xd["weight"], qd, xd["targets"], None,
                                    w.ignore_index, 1.0, 1e-10, "batchmean", err_word=err,
                                    skip_ignored=True)
    go = torch.tensor(1.0, dtype=torch.float32, device="cuda")
    gh, gw, _ = api.flce_kl_backward_tensors(xd["hidden"], xd["weight"], qd, f["lse_rows"],
                                             f["qsum_rows"], f["n_counted"], go, xd["targets"],
                                             None, w.ignore_index, 1.0, 1e-10, "batchmean",
                                             err_word=err, skip_ignored=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    del qd
    ref = kl_oracle.forward(x["hidden"], x["weight"], q, None, x["targets"], w.ignore_index, 1.0,
                            1e-10, "batchmean")
    counted = ref["counted"]
    assert int(f["n_counted"]) == ref["n_counted"]
    floor = row_floor(w.h, kl_row_ops(ref))
    assert_rows_close("loss_rows", f["loss_rows"].cpu(), ref["loss"], tol["loss_rel"],
                      floor=floor)
    assert_rows_close("lse_rows", f["lse_rows"].cpu(), ref["lse"], tol["loss_rel"], counted,
                      floor)
    assert_rows_close("qsum_rows", f["qsum_rows"].cpu(), ref["qsum"], 1e-5, counted)
    nc = ref["n_counted"]
    assert_scalar_close("loss", float(f["loss"]), ref["loss_out"], tol["loss_rel"],
                        float(floor[counted].sum()) / nc,
                        float(ref["loss"][counted].abs().sum()) / nc, nc)
    rows = _sample_rows(w, x["targets"], torch.empty(0, dtype=torch.int64), k=256)
    vocab = _sample_vocab(w, x["targets"], rows, torch.empty(0, dtype=torch.int64), k=128)
    gref = kl_oracle.backward(x["hidden"], x["weight"], q, None, x["targets"], w.ignore_index,
                              1.0, 1e-10, "batchmean", 1.0, rows=rows, vocab_rows=vocab,
                              magnitudes=True)
    gh_c, gw_c = gh.cpu(), gw.cpu()
    kap = grad_kappas(w)
    assert_grad_close("grad_hidden", gh_c[rows], gref["grad_hidden"], tol,
                      gref["grad_hidden_mag"], kap["grad_hidden"])
    assert_grad_close("grad_weight", gw_c[vocab], gref["grad_weight"], tol,
                      gref["grad_weight_mag"], kap["grad_weight"])
    assert torch.all(gh_c[~counted] == 0)
    g64 = gw_c.double()
    col = g64.sum(dim=0).abs()
    mag = g64.abs().sum(dim=0)
    assert bool((col <= 1e-2 * mag + 1e-12).all()), float((col / mag).max())


@pytest.mark.parametrize("name,kl", [("llama3_head_bf16", False), ("llama3_head_bf16", True),
                                     ("mid_bf16", False), ("softcap_bf16", False),
                                     ("long_bf16", False)])
def test_peak_memory_below_logits(name, kl):
    """One forward+backward through the public autograd API, with the
    workload's options and the library's default chunking, allocates above
    what is live before it (inputs, and the teacher probabilities for KL)
    less than the N x V logit matrix would take in bf16 (N*V*2 bytes): the
    logits are never materialised. The incremental peak includes grad_weight
    [V, H], grad_hidden, grad_bias and the workspaces. At the mid shape
    grad_weight alone is half of N*V*2, so this also pins the default
    chunking's fifth-of-the-vocabulary bound."""
    from linear_cross_entropy_vocab_gb300 import fused_linear_cross_entropy, fused_linear_kl_div
    from linear_cross_entropy_vocab_gb300.workloads import make_teacher_probs

    w = WORKLOADS[name]
    x = to_dev(make_inputs(w))
    q = make_teacher_probs(w).cuda() if kl else None
    h = x["hidden"].detach().requires_grad_(True)
    wt = x["weight"].detach().requires_grad_(True)
    b = None if x["bias"] is None else x["bias"].detach().requires_grad_(True)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    if kl:
        loss = fused_linear_kl_div(h, wt, q, x["targets"])
    else:
        loss = fused_linear_cross_entropy(h, wt, x["targets"], b, w.ignore_index, w.logit_scale,
                                          w.softcap, w.reduction)
    loss.backward()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    nxv = w.n * w.v * 2
    assert peak < nxv, (peak, nxv)
    assert torch.isfinite(loss).item()


def test_largest_vocabulary_sampled():
    """A 262144-entry vocabulary (1024 vocabulary tiles per row; 8 backward
    chunks), N=4096, H=2048, bf16, bias and softcap, 10 % ignored rows left
    out: every row's loss and lse against the oracle, gradients on sampled
    rows and vocabulary entries."""
    w = Workload("v262144", 4096, 2048, 262144, "bf16", bias_var=0.02, softcap=30.0,
                 logit_scale=0.9, ignore_frac=0.1, reduction="mean")
    x = make_inputs(w)
    xd = to_dev(x)
    tol = TOL[w.dtype]
    out = run_gpu(xd, w, grad_out=1.0, skip_ignored=True, row_metrics=True)
    assert out["err_word"] == 0
    ref = oracle.forward(*oracle_args(x, w))
    check_forward(out, ref, w, tol, skipped=True)
    rows = _sample_rows(w, x["targets"], torch.empty(0, dtype=torch.int64), k=128)
    vocab = _sample_vocab(w, x["targets"], rows, torch.empty(0, dtype=torch.int64), k=128)
    gref = oracle.backward(*oracle_args(x, w), 1.0, lse=ref["lse"], rows=rows, vocab_rows=vocab,
                           magnitudes=True)
    sampled = {"grad_hidden": out["grad_hidden"][rows], "grad_weight": out["grad_weight"][vocab],
               "grad_bias": out["grad_bias"][vocab]}
    check_backward(sampled, gref, tol, True, grad_kappas(w))
