"""Host-side checks of the C ABI, runnable without a GPU: the library builds,
loads and exports every function include/flce.h declares; the ctypes struct
matches the C struct; workspace sizing; and argument validation, which
returns its status before any CUDA call (no kernel is launched here)."""
import ctypes
import os
import re

import pytest

from linear_cross_entropy_vocab_gb300 import abi, native_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")


@pytest.fixture(scope="module")
def lib():
    native_build.build()
    return abi.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flce_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert declared == sorted(abi.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_struct_layout_matches_header():
    # int64 n,h,v; int32 dtype,has_bias; int64 ignore_index; float scale, softcap;
    # int32 reduction, grad_weight_dtype; int64 vocab_chunk; int32 flags;
    # float label_smoothing, z_loss; int32 reserved
    assert ctypes.sizeof(abi.flce_problem) == 80
    assert abi.flce_problem.ignore_index.offset == 32
    assert abi.flce_problem.logit_scale.offset == 40
    assert abi.flce_problem.vocab_chunk.offset == 56
    assert abi.flce_problem.flags.offset == 64
    assert abi.flce_problem.z_loss.offset == 72


def test_status_strings(lib):
    assert abi.flce_status_string(abi.FLCE_OK) == "FLCE_OK"
    assert abi.flce_status_string(abi.FLCE_ERR_WORKSPACE) == "FLCE_ERR_WORKSPACE"


def test_workspace_sizes(lib):
    p = abi.make_problem(8192, 4096, 128256, abi.FLCE_BF16, False)
    fwd = abi.flce_forward_workspace_size(p)
    # per-(row, 256-wide vocabulary tile) statistics: 16 bytes each
    assert fwd >= 8192 * 501 * 16
    assert fwd < 8192 * 128256 * 2 // 16  # far below the N x V logits
    bwd = abi.flce_backward_workspace_size(p)
    assert bwd < 8192 * 128256 * 2  # never N x V in bf16
    p.vocab_chunk = 1000
    small = abi.flce_backward_workspace_size(p)
    assert small >= 8192 * 1024 * 2  # rounded up to a multiple of 256
    bad = abi.make_problem(8, 12, 100, abi.FLCE_BF16, False)  # h % 8 != 0
    assert abi.flce_forward_workspace_size(bad) == 0


FAKE = 0x10000  # never dereferenced: validation fails before any device access


def _fwd(p, **kw):
    args = dict(hidden=FAKE, weight=FAKE, bias=None, targets=FAKE, loss_rows=FAKE,
                lse_rows=FAKE, correct_rows=None, entropy_rows=None, loss_out=FAKE,
                metrics_out=None, n_valid=FAKE, err_word=None, workspace=FAKE,
                workspace_bytes=1 << 40, stream=None)
    args.update(kw)
    return abi.flce_forward(p, check=False, **args)


def _bwd(p, **kw):
    args = dict(hidden=FAKE, weight=FAKE, bias=None, targets=FAKE, lse_rows=FAKE,
                n_valid=FAKE, grad_out=FAKE, grad_hidden=FAKE, grad_weight=FAKE,
                grad_bias=None, err_word=None, workspace=FAKE, workspace_bytes=1 << 40,
                stream=None)
    args.update(kw)
    return abi.flce_backward(p, check=False, **args)


def test_validation_statuses(lib):
    ok = abi.make_problem(64, 64, 100, abi.FLCE_BF16, False)
    assert _fwd(ok, weight=None) == abi.FLCE_ERR_INVALID_ARG
    assert _fwd(ok, n_valid=None) == abi.FLCE_ERR_INVALID_ARG
    assert _fwd(ok, loss_out=None) == abi.FLCE_ERR_INVALID_ARG  # mean needs loss_out
    assert _fwd(ok, bias=FAKE) == abi.FLCE_ERR_INVALID_ARG  # bias without has_bias
    assert _fwd(ok, hidden=FAKE + 2) == abi.FLCE_ERR_UNSUPPORTED  # misaligned
    assert _fwd(ok, workspace_bytes=16) == abi.FLCE_ERR_WORKSPACE
    assert _fwd(ok, workspace=FAKE + 8) == abi.FLCE_ERR_WORKSPACE  # not 256-aligned
    assert "workspace" in abi.flce_last_error()
    neg = abi.make_problem(-1, 64, 100, abi.FLCE_BF16, False)
    assert _fwd(neg) == abi.FLCE_ERR_INVALID_ARG
    odd = abi.make_problem(64, 60, 100, abi.FLCE_BF16, False)
    assert _fwd(odd) == abi.FLCE_ERR_UNSUPPORTED
    red = abi.make_problem(64, 64, 100, abi.FLCE_BF16, False)
    red.reduction = 7
    assert _fwd(red) == abi.FLCE_ERR_INVALID_ARG
    cap = abi.make_problem(64, 64, 100, abi.FLCE_BF16, False, softcap=float("nan"))
    assert _fwd(cap) == abi.FLCE_ERR_INVALID_ARG
    gw = abi.make_problem(64, 64, 100, abi.FLCE_F32, False, grad_weight_dtype=abi.FLCE_BF16)
    assert _fwd(gw) == abi.FLCE_ERR_INVALID_ARG
    ls = abi.make_problem(64, 64, 100, abi.FLCE_BF16, False, label_smoothing=1.5)
    assert _fwd(ls) == abi.FLCE_ERR_INVALID_ARG
    zl = abi.make_problem(64, 64, 100, abi.FLCE_BF16, False, z_loss=float("inf"))
    assert _fwd(zl) == abi.FLCE_ERR_INVALID_ARG
    none = abi.make_problem(64, 64, 100, abi.FLCE_BF16, False, reduction="none")
    assert _fwd(none, loss_out=None, workspace_bytes=8) == abi.FLCE_ERR_WORKSPACE
    bias = abi.make_problem(64, 64, 100, abi.FLCE_BF16, True)
    assert _bwd(bias) == abi.FLCE_ERR_INVALID_ARG  # bias and grad_bias missing
    assert _bwd(ok, grad_out=None) == abi.FLCE_ERR_INVALID_ARG
    assert _bwd(ok, grad_hidden=FAKE + 4) == abi.FLCE_ERR_UNSUPPORTED
    assert _bwd(ok, workspace_bytes=0) == abi.FLCE_ERR_WORKSPACE
    assert lib.flce_forward(None, *([None] * 13), 0, None) == abi.FLCE_ERR_INVALID_ARG


def _c_layout():
    """sizeof / offsetof of both problem structs as a C compiler lays them
    out from include/flce.h (gcc on this host)."""
    import shutil
    import subprocess
    import tempfile
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = r"""
#include <stddef.h>
#include <stdio.h>
#include "flce.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu\n", sizeof(flce_problem), offsetof(flce_problem, ignore_index),
         offsetof(flce_problem, logit_scale), offsetof(flce_problem, flags),
         offsetof(flce_problem, z_loss));
  printf("%zu %zu %zu %zu %zu\n", sizeof(flce_kl_problem),
         offsetof(flce_kl_problem, ignore_index), offsetof(flce_kl_problem, temperature),
         offsetof(flce_kl_problem, vocab_chunk), offsetof(flce_kl_problem, reserved));
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe],
                       check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split("\n")
    return [int(x) for x in out[0].split()], [int(x) for x in out[1].split()]


def test_struct_layouts_match_c_compiler():
    ce, kl = _c_layout()
    P, K = abi.flce_problem, abi.flce_kl_problem
    assert ce == [ctypes.sizeof(P), P.ignore_index.offset, P.logit_scale.offset,
                  P.flags.offset, P.z_loss.offset]
    assert kl == [ctypes.sizeof(K), K.ignore_index.offset, K.temperature.offset,
                  K.vocab_chunk.offset, K.reserved.offset]
    assert ctypes.sizeof(K) == 72


def _kl_fwd(p, **kw):
    args = dict(hidden=FAKE, weight=FAKE, bias=None, target_probs=FAKE, labels=None,
                loss_rows=FAKE, lse_rows=FAKE, qsum_rows=FAKE, loss_out=FAKE, n_counted=FAKE,
                err_word=None, workspace=FAKE, workspace_bytes=1 << 40, stream=None)
    args.update(kw)
    return abi.flce_kl_forward(p, check=False, **args)


def _kl_bwd(p, **kw):
    args = dict(hidden=FAKE, weight=FAKE, bias=None, target_probs=FAKE, labels=None,
                lse_rows=FAKE, qsum_rows=FAKE, n_counted=FAKE, grad_out=FAKE,
                grad_hidden=FAKE, grad_weight=FAKE, grad_bias=None, err_word=None,
                workspace=FAKE, workspace_bytes=1 << 40, stream=None)
    args.update(kw)
    return abi.flce_kl_backward(p, check=False, **args)


def test_kl_validation_and_workspace(lib):
    ok = abi.make_kl_problem(64, 64, 100, abi.FLCE_BF16, False)
    assert abi.flce_kl_forward_workspace_size(ok) >= 64 * 1 * 16
    big = abi.make_kl_problem(8192, 4096, 128256, abi.FLCE_BF16, False)
    assert abi.flce_kl_backward_workspace_size(big) < 8192 * 128256 * 2
    for field, bad in (("temperature", 0.0), ("temperature", float("nan")),
                       ("temperature", -1.0), ("temperature", 1e-39), ("eps", 0.0),
                       ("eps", float("inf")), ("reduction", 4), ("reserved", 1)):
        p = abi.make_kl_problem(64, 64, 100, abi.FLCE_BF16, False)
        setattr(p, field, bad)
        assert _kl_fwd(p) == abi.FLCE_ERR_INVALID_ARG, field
        assert abi.flce_kl_forward_workspace_size(p) == 0
    assert _kl_fwd(ok, target_probs=None) == abi.FLCE_ERR_INVALID_ARG
    assert _kl_fwd(ok, qsum_rows=None) == abi.FLCE_ERR_INVALID_ARG
    assert _kl_fwd(ok, n_counted=None) == abi.FLCE_ERR_INVALID_ARG
    assert _kl_fwd(ok, loss_out=None) == abi.FLCE_ERR_INVALID_ARG  # batchmean needs it
    assert _kl_fwd(ok, target_probs=FAKE + 1) == abi.FLCE_ERR_UNSUPPORTED
    assert _kl_fwd(ok, labels=FAKE + 4) == abi.FLCE_ERR_UNSUPPORTED
    assert _kl_fwd(ok, workspace_bytes=16) == abi.FLCE_ERR_WORKSPACE
    odd = abi.make_kl_problem(64, 60, 100, abi.FLCE_BF16, False)
    assert _kl_fwd(odd) == abi.FLCE_ERR_UNSUPPORTED
    assert _kl_bwd(ok, target_probs=None) == abi.FLCE_ERR_INVALID_ARG
    assert _kl_bwd(ok, qsum_rows=None) == abi.FLCE_ERR_INVALID_ARG
    assert _kl_bwd(ok, grad_out=None) == abi.FLCE_ERR_INVALID_ARG
    assert _kl_bwd(ok, workspace_bytes=0) == abi.FLCE_ERR_WORKSPACE
    assert lib.flce_kl_forward(None, *([None] * 12), 0, None) == abi.FLCE_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["tiny_fp32", "mid_bf16", "llama3_head_bf16", "softcap_bf16",
                                  "long_bf16"])
@pytest.mark.parametrize("as_f32", [False, True])
def test_planned_peak_below_logits(lib, name, as_f32):
    """The host plan behind the no-N x V guarantee: the larger of the two
    workspaces plus the gradients a step returns (grad_weight [V, H],
    grad_hidden [N, H], grad_bias [V]) stay under one N x V logit matrix in
    the input type, for every listed workload in its own type and in fp32
    (where the split path adds the operands' bf16 parts and D's three parts).
    The GPU test of peak allocation measures the same bound on the device;
    this pins the sizing on the host, so that a larger default chunk or a
    new workspace region that would break it fails without a GPU."""
    from linear_cross_entropy_vocab_gb300.workloads import WORKLOADS

    w = WORKLOADS[name]
    dt = abi.FLCE_F32 if (as_f32 or w.dtype == "f32") else abi.FLCE_BF16
    el = 4 if dt == abi.FLCE_F32 else 2
    has_bias = w.bias_var is not None
    p = abi.make_problem(w.n, w.h, w.v, dt, has_bias, skip_ignored=True)
    ws = max(abi.flce_forward_workspace_size(p), abi.flce_backward_workspace_size(p))
    k = abi.make_kl_problem(w.n, w.h, w.v, dt, False, skip_ignored=True)
    wk = max(abi.flce_kl_forward_workspace_size(k), abi.flce_kl_backward_workspace_size(k))
    assert ws > 0 and wk > 0
    grads = (w.v * w.h + w.n * w.h) * el
    logits = w.n * w.v * el
    assert ws + grads + (w.v * el if has_bias else 0) < logits, (ws, grads, logits)
    assert wk + grads < logits, (wk, grads, logits)
