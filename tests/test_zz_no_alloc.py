"""flce_forward_noalloc: the forward pass for callers that cannot allocate
device memory (for example a host framework whose memory pool owns the whole
GPU and refuses allocations from libraries, or a latency-bound loop where a
cudaMalloc, which may synchronise the device, is not allowed) and so have no
workspace to hand to flce_forward. Its scratch is a fixed 16 MiB array inside
the library.

The GPU tests call it through the C ABI several times in a row, on different
problems, and check each result against flce_forward's on the same inputs
within the parity tolerances of tests/_parity.py, and against the fp64
oracle. Every call after the first runs on scratch that still holds an
earlier call's contents; the cases with FLCE_SKIP_IGNORED_ROWS and label
smoothing use the scratch regions (row map, kept-row count, gathered rows and
targets, per-tile logit sums) that the plain forward leaves untouched. This
file is named so that pytest collects it last.
"""
import pytest
import torch

import oracle
from _parity import (TOL, assert_rows_close, assert_scalar_close, ce_row_ops, check_forward,
                     oracle_args, oracle_opts, row_floor)
from linear_cross_entropy_vocab_gb300 import abi, api, native_build
from linear_cross_entropy_vocab_gb300.workloads import Workload, make_inputs

STATIC_SCRATCH_BYTES = 16 << 20


def _problem(w, n, h, v, dtype, has_bias, skip):
    return abi.make_problem(n, h, v, dtype, has_bias, w.ignore_index, w.logit_scale, w.softcap,
                            w.reduction, skip_ignored=skip, label_smoothing=w.label_smoothing,
                            z_loss=w.z_loss)


def _noalloc_forward(xd, w, skip=False, metrics=True):
    """One flce_forward_noalloc call; with metrics=False the per-row
    correctness, per-row entropy and metrics outputs are NULL."""
    n, h = xd["hidden"].shape
    v = xd["weight"].shape[0]
    dev = xd["hidden"].device
    dtype = abi.FLCE_BF16 if xd["hidden"].dtype == torch.bfloat16 else abi.FLCE_F32
    prob = _problem(w, n, h, v, dtype, xd["bias"] is not None, skip)
    assert abi.flce_forward_workspace_size(prob) <= STATIC_SCRATCH_BYTES
    f32 = dict(dtype=torch.float32, device=dev)
    out = {
        "loss_rows": torch.empty(n, **f32), "lse_rows": torch.empty(n, **f32),
        "correct_rows": torch.empty(n, dtype=torch.int32, device=dev) if metrics else None,
        "entropy_rows": torch.empty(n, **f32) if metrics else None,
        "loss": torch.empty((), **f32),
        "metrics": torch.empty(2, **f32) if metrics else None,
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
    return {k: (None if t is None else t.cpu()) for k, t in out.items()}


def _same(a, b):
    """Bitwise equal, NaN where the other is NaN."""
    return torch.equal(torch.isnan(a), torch.isnan(b)) and torch.equal(
        a[~torch.isnan(a)], b[~torch.isnan(b)])


def _workspace_forward(xd, w, skip=False):
    ref = api.flce_forward_tensors(xd["hidden"], xd["weight"], xd["targets"], xd["bias"],
                                   w.ignore_index, w.logit_scale, w.softcap, w.reduction,
                                   return_metrics=True, row_metrics=True, skip_ignored=skip,
                                   label_smoothing=w.label_smoothing, z_loss=w.z_loss)
    return {k: (None if t is None else t.cpu()) for k, t in ref.items()}


def _compare_with_workspace_forward(got, ref, metrics=True):
    """The same kernels run on the same inputs, so the results are bitwise
    flce_forward's (the per-row loss and lse do not depend on whether the
    metric outputs are requested)."""
    assert int(got["n_valid"]) == int(ref["n_valid"])
    for k in ("loss_rows", "lse_rows", "loss"):
        assert _same(got[k], ref[k]), k
    if metrics:
        for k in ("entropy_rows", "metrics", "correct_rows"):
            assert _same(got[k], ref[k]), k


def _compare_with_oracle(got, x, w, skip):
    ref = oracle.forward(*oracle_args(x, w), **oracle_opts(w))
    check_forward(got, ref, w, TOL[w.dtype], skipped=skip)


def _run(w, skip=False, metrics=True):
    x = make_inputs(w)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    got = _noalloc_forward(xd, w, skip=skip, metrics=metrics)
    _compare_with_workspace_forward(got, _workspace_forward(xd, w, skip), metrics)
    return got, x


@pytest.mark.gpu
def test_noalloc_forward_matches_workspace_forward_twice():
    native_build.build()
    cases = [
        Workload("noalloc_a", 1500, 1024, 32000, "bf16", bias_var=0.02, ignore_frac=0.1,
                 softcap=30.0, logit_scale=0.7, reduction="mean"),
        Workload("noalloc_b", 777, 512, 9001, "bf16", ignore_frac=0.05, reduction="sum"),
    ]
    for w in cases:
        _run(w)


@pytest.mark.gpu
def test_noalloc_skip_ignored_label_smoothing_after_a_larger_call():
    """A larger plain call first fills the scratch; then a call with
    FLCE_SKIP_IGNORED_ROWS and label smoothing, whose row map, kept-row count,
    gathered rows and per-tile logit sums sit in scratch that the first call
    wrote with other contents. Checked against flce_forward and the oracle."""
    native_build.build()
    big = Workload("noalloc_big", 1800, 1024, 32000, "bf16", bias_var=0.02, ignore_frac=0.1,
                   reduction="mean")
    _run(big)
    w = Workload("noalloc_skip_ls", 600, 1024, 32000, "bf16", bias_var=0.02, ignore_frac=0.1,
                 label_smoothing=0.1, reduction="mean", return_metrics=True)
    got, x = _run(w, skip=True)
    _compare_with_oracle(got, x, w, skip=True)
    # and once more right after it, on a problem that skips no row
    w2 = Workload("noalloc_skip_ls_b", 333, 512, 5000, "bf16", ignore_frac=0.0,
                  label_smoothing=0.2, z_loss=1e-3, reduction="sum", return_metrics=True)
    got2, x2 = _run(w2, skip=True)
    _compare_with_oracle(got2, x2, w2, skip=True)


@pytest.mark.gpu
def test_noalloc_without_metrics_outputs():
    """correct_rows, entropy_rows and metrics_out NULL: the forward skips the
    argmax and entropy terms; loss, lse and n_valid match the oracle."""
    native_build.build()
    w = Workload("noalloc_nometrics", 900, 512, 20000, "bf16", ignore_frac=0.05,
                 softcap=20.0, logit_scale=0.8, reduction="sum")
    got, x = _run(w, metrics=False)
    ref = oracle.forward(*oracle_args(x, w), **oracle_opts(w))
    tol = TOL[w.dtype]
    nv = ref["n_valid"]
    assert int(got["n_valid"]) == nv
    floor = row_floor(w.h, ce_row_ops(ref))
    assert_rows_close("loss_rows", got["loss_rows"], ref["loss"], tol["loss_rel"], floor=floor)
    assert_rows_close("lse_rows", got["lse_rows"], ref["lse"], tol["loss_rel"], floor=floor)
    valid = ref["valid"]
    assert_scalar_close("loss", float(got["loss"]), ref["loss_out"], tol["loss_rel"],
                        float(floor[valid].sum()), float(ref["loss"][valid].abs().sum()), nv)


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


def test_noalloc_reports_what_flce_forward_reports():
    """Argument errors come first in both entry points, and on a host whose
    current device is absent or not sm_103a both return the same status and
    message for the same valid call (the device is checked before the
    scratch's address is looked up). Pointers are never dereferenced: every
    call returns before any launch."""
    native_build.build()
    if abi.flce_device_supported():
        pytest.skip("a supported GPU is present: the call would run")
    prob = abi.make_problem(256, 64, 1000, abi.FLCE_BF16, False)
    fake = 0x10000
    ws = abi.flce_forward_workspace_size(prob)
    st_ws = abi.flce_forward(prob, fake, fake, None, fake, fake, fake, None, None, fake, None,
                             fake, None, fake, ws, None, check=False)
    msg_ws = abi.flce_last_error()
    st_na = abi.flce_forward_noalloc(prob, fake, fake, None, fake, fake, fake, None, None, fake,
                                     None, fake, None, None, check=False)
    msg_na = abi.flce_last_error()
    assert st_ws != abi.FLCE_OK
    assert (st_na, msg_na) == (st_ws, msg_ws)
    # a missing required pointer is an argument error in both, before the device
    st_ws = abi.flce_forward(prob, None, fake, None, fake, fake, fake, None, None, fake, None,
                             fake, None, fake, ws, None, check=False)
    st_na = abi.flce_forward_noalloc(prob, None, fake, None, fake, fake, fake, None, None, fake,
                                     None, fake, None, None, check=False)
    assert st_ws == st_na == abi.FLCE_ERR_INVALID_ARG
