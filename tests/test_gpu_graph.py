"""CUDA-graph capture of a whole training step.

The forward and backward entry points only enqueue work on the caller's
stream: they never wait on the host, never read device values on the host
(the kept-row count of the row compaction is read by the kernels themselves)
and allocate nothing (the caller passes the workspace). So one forward +
backward can be captured into a CUDA graph once and replayed with new inputs
copied into the captured buffers; every replay must give bitwise the results
of eager calls on the same inputs, including a different number of ignored
rows from one replay to the next.
"""
import dataclasses

import pytest
import torch

from _parity import to_dev
from linear_cross_entropy_vocab_gb300 import api
from linear_cross_entropy_vocab_gb300.workloads import Workload, make_inputs, make_teacher_probs

pytestmark = pytest.mark.gpu


def _ce_step(x, w, go, skip):
    f = api.flce_forward_tensors(x["hidden"], x["weight"], x["targets"], x["bias"],
                                 w.ignore_index, w.logit_scale, w.softcap, w.reduction,
                                 return_metrics=True, row_metrics=True, skip_ignored=skip,
                                 vocab_chunk=w.v // 3)
    gh, gw, gb = api.flce_backward_tensors(x["hidden"], x["weight"], x["targets"],
                                           f["lse_rows"], f["n_valid"], go, x["bias"],
                                           w.ignore_index, w.logit_scale, w.softcap,
                                           w.reduction, skip_ignored=skip,
                                           vocab_chunk=w.v // 3)
    return {"loss": f["loss"], "loss_rows": f["loss_rows"], "metrics": f["metrics"],
            "n_valid": f["n_valid"], "correct_rows": f["correct_rows"], "grad_hidden": gh,
            "grad_weight": gw, "grad_bias": gb}


def _kl_step(x, w, go, skip):
    f = api.flce_kl_forward_tensors(x["hidden"], x["weight"], x["q"], x["targets"], x["bias"],
                                    w.ignore_index, temperature=1.5, reduction="batchmean",
                                    skip_ignored=skip)
    gh, gw, gb = api.flce_kl_backward_tensors(x["hidden"], x["weight"], x["q"], f["lse_rows"],
                                              f["qsum_rows"], f["n_counted"], go,
                                              x["targets"], x["bias"], w.ignore_index,
                                              temperature=1.5, reduction="batchmean",
                                              skip_ignored=skip, vocab_chunk=w.v // 3)
    return {"loss": f["loss"], "loss_rows": f["loss_rows"], "n_counted": f["n_counted"],
            "grad_hidden": gh, "grad_weight": gw, "grad_bias": gb}


def _inputs(w, kl):
    x = make_inputs(w)
    if kl:
        x["q"] = make_teacher_probs(w)
    return to_dev(x)


CASES = [
    ("bf16", False, False),
    ("bf16", True, False),
    ("f16", True, False),
    ("f32", False, False),
    ("bf16", True, True),
]


@pytest.mark.parametrize("dtype,skip,kl", CASES,
                         ids=[f"{d}-{'skip' if s else 'all'}-{'kl' if k else 'ce'}"
                              for d, s, k in CASES])
def test_captured_step_replays_bitwise(dtype, skip, kl):
    w = Workload("graph", 700, 192, 5000, dtype, bias_var=0.02, softcap=None if kl else 25.0,
                 ignore_frac=0.1)
    step = _kl_step if kl else _ce_step
    x = _inputs(w, kl)  # the captured buffers
    go = torch.tensor(0.75, dtype=torch.float32, device="cuda")

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one-time library set-up happens outside the capture
        for _ in range(2):
            step(x, w, go, skip)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = step(x, w, go, skip)

    # new inputs each replay: other values and another set (and count) of ignored rows
    for seed, frac in ((1, 0.05), (2, 0.3)):
        nxt = _inputs(dataclasses.replace(w, seed=seed, ignore_frac=frac), kl)
        for k, t in nxt.items():
            if t is not None:
                x[k].copy_(t)
        graph.replay()
        ref = step(x, w, go, skip)
        torch.cuda.synchronize()
        for k, v in ref.items():
            if v is None:
                assert out[k] is None
                continue
            assert torch.equal(out[k], v), k
        n_kept = out["n_counted" if kl else "n_valid"]
        assert int(n_kept) == int((nxt["targets"] != w.ignore_index).sum())
