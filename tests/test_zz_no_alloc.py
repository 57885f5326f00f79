"""flce_forward_noalloc: the forward pass for callers that cannot allocate
device memory (for example a host framework whose memory pool owns the whole
GPU and refuses allocations from libraries, or a latency-bound loop where a
cudaMalloc, which may synchronise the device, is not allowed) and so have no
workspace to hand to flce_forward. Its scratch is a fixed 16 MiB array inside
the library.

The GPU test calls it through the C ABI twice in a row, on two different
problems, and checks each result against flce_forward's on the same inputs
within the parity tolerances of tests/_parity.py. The second call runs on
scratch that still holds the first call's contents. This file is named so
that pytest collects it last.
"""
import ctypes

import pytest
import torch

from _parity import TOL
from linear_cross_entropy_vocab_gb300 import abi, api, native_build
from linear_cross_entropy_vocab_gb300.workloads import Workload, make_inputs

STATIC_SCRATCH_BYTES = 16 << 20


def _noalloc_forward(xd, w):
    n, h = xd["hidden"].shape
    v = xd["weight"].shape[0]
    dev = xd["hidden"].device
    dtype = abi.FLCE_BF16 if xd["hidden"].dtype == torch.bfloat16 else abi.FLCE_F32
    prob = abi.make_problem(n, h, v, dtype, xd["bias"] is not None, w.ignore_index,
                            w.logit_scale, w.softcap, w.reduction)
    f32 = dict(dtype=torch.float32, device=dev)
    out = {
        "loss_rows": torch.empty(n, **f32), "lse_rows": torch.empty(n, **f32),
        "correct_rows": torch.empty(n, dtype=torch.int32, device=dev),
        "entropy_rows": torch.empty(n, **f32), "loss": torch.empty((), **f32),
        "metrics": torch.empty(2, **f32),
        "n_valid": torch.empty((), dtype=torch.int32, device=dev),
    }
    err = torch.zeros((), dtype=torch.int32, device=dev)
    p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    abi.flce_forward_noalloc(prob, p(xd["hidden"]), p(xd["weight"]), p(xd["bias"]),
                             p(xd["targets"]), p(out["loss_rows"]), p(out["lse_rows"]),
                             p(out["correct_rows"]), p(out["entropy_rows"]), p(out["loss"]),
                             p(out["metrics"]), p(out["n_valid"]), p(err),
                             torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0
    return {k: t.cpu() for k, t in out.items()}


def _close(a, b, rel):
    a, b = a.double(), b.double()
    return bool(((a - b).abs() <= rel * b.abs().clamp_min(1.0)).all())


@pytest.mark.gpu
def test_noalloc_forward_matches_workspace_forward_twice():
    native_build.build()
    cases = [
        Workload("noalloc_a", 1500, 1024, 32000, "bf16", bias_var=0.02, ignore_frac=0.1,
                 softcap=30.0, logit_scale=0.7, reduction="mean"),
        Workload("noalloc_b", 777, 512, 9001, "bf16", ignore_frac=0.05, reduction="sum"),
    ]
    for w in cases:
        x = make_inputs(w)
        xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
        prob = abi.make_problem(w.n, w.h, w.v, abi.FLCE_BF16, w.bias_var is not None)
        assert abi.flce_forward_workspace_size(prob) <= STATIC_SCRATCH_BYTES
        got = _noalloc_forward(xd, w)
        ref = api.flce_forward_tensors(xd["hidden"], xd["weight"], xd["targets"], xd["bias"],
                                       w.ignore_index, w.logit_scale, w.softcap, w.reduction,
                                       return_metrics=True, row_metrics=True)
        ref = {k: (None if t is None else t.cpu()) for k, t in ref.items()}
        tol = TOL[w.dtype]
        assert int(got["n_valid"]) == int(ref["n_valid"])
        assert _close(got["loss_rows"], ref["loss_rows"], tol["loss_rel"])
        assert _close(got["lse_rows"], ref["lse_rows"], tol["loss_rel"])
        assert _close(got["entropy_rows"], ref["entropy_rows"], tol["ent_rel"])
        assert _close(got["loss"], ref["loss"], tol["loss_rel"])
        assert _close(got["metrics"], ref["metrics"], tol["ent_rel"])
        assert torch.equal(got["correct_rows"], ref["correct_rows"])


def test_noalloc_rejects_problems_beyond_the_fixed_scratch():
    """Rejected on the host before any device work (no GPU needed)."""
    native_build.build()
    big = abi.make_problem(8192, 4096, 128256, abi.FLCE_BF16, False)
    assert abi.flce_forward_workspace_size(big) > STATIC_SCRATCH_BYTES
    fake = 0x10000  # never dereferenced: the size check fails first
    st = abi.flce_forward_noalloc(big, fake, fake, None, fake, fake, fake, None, None, fake,
                                  None, fake, None, None, check=False)
    assert st == abi.FLCE_ERR_UNSUPPORTED
    assert "fixed scratch" in abi.flce_last_error()
