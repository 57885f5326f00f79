"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle,
element by element, at sizes the oracle finishes in seconds. The shapes cover
several tiles with a ragged tail along each of N (tokens), V (vocabulary) and
H (hidden), multi-chunk backward passes, every option of the kernel card's
signature, and the degenerate cases.

Tolerances are documented in ``tests/_parity.py``.
"""
import math

import pytest
import torch

import oracle
from _parity import (TOL, assert_grad_close, assert_rows_close, check_backward, check_forward,
                     ce_row_ops, grad_kappas, oracle_args, oracle_opts, row_floor, run_gpu,
                     to_dev)
from linear_cross_entropy_vocab_gb300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


def _case(name, n, h, v, dtype="bf16", **kw):
    return Workload(name, n, h, v, dtype, **kw)


CASES = [
    # the small fp32 workload exactly as specified (N=256, H=128, V=1000)
    WORKLOADS["tiny_fp32"],
    # ragged N (300 = 2*128+44), V (1000 = 3*256+232) and H (136 = 2*64+8)
    _case("tails_bias_cap_sum", 300, 136, 1000, bias_var=0.02, softcap=30.0,
          logit_scale=0.5, hidden_var=2.0, ignore_frac=0.3, reduction="sum"),
    _case("v32003_mean", 512, 256, 32003, ignore_frac=0.05),
    _case("n4097_none", 4097, 512, 4096, ignore_frac=0.1, reduction="none"),
    _case("h3592_cap", 256, 3592, 2048, softcap=30.0, logit_scale=0.5, hidden_var=2.0,
          ignore_frac=0.3, reduction="sum"),
    # H > 2048 runs the relayed 4-warp epilogues; ragged N, H and V, metrics on
    _case("h2312_relay_bias", 300, 2312, 1000, bias_var=0.02, ignore_frac=0.1,
          return_metrics=True),
    # the relay with a single row, and with a last vocabulary tile of one column (the
    # computing warps take one chunk and release the other seven unread)
    _case("relay_n1", 1, 2112, 777, bias_var=0.02, return_metrics=True),
    _case("relay_v513_none", 129, 2112, 513, ignore_frac=0.1, reduction="none"),
    _case("v152063", 256, 128, 152063, ignore_frac=0.02, return_metrics=True),
    _case("zipf_bias_mean", 640, 192, 5000, bias_var=0.02, targets="zipf", ignore_frac=0.1),
    _case("peaked_rows", 384, 256, 3000, peaked_frac=0.01, ignore_frac=0.05),
    _case("f32_cap_none", 100, 50, 777, dtype="f32", bias_var=0.02, softcap=5.0,
          logit_scale=1.5, ignore_frac=0.1, reduction="none"),
    _case("f32_sum_bias", 257, 96, 2100, dtype="f32", bias_var=0.5, reduction="sum"),
]


def _grad_out(w, n):
    if w.reduction == "none":
        g = torch.Generator().manual_seed(7)
        return torch.rand(n, generator=g, dtype=torch.float64) + 0.5
    return 0.75


def _check_case(w, vocab_chunk=0, grad_weight_dtype=None, skip_ignored=False):
    x = make_inputs(w)
    go = _grad_out(w, w.n)
    out = run_gpu(to_dev(x), w, grad_out=go.float() if torch.is_tensor(go) else go,
                  vocab_chunk=vocab_chunk, grad_weight_dtype=grad_weight_dtype,
                  skip_ignored=skip_ignored)
    assert out["err_word"] == 0
    ref = oracle.forward(*oracle_args(x, w), **oracle_opts(w))
    tol = TOL[w.dtype]
    check_forward(out, ref, w, tol, skipped=skip_ignored and w.dtype != "f32")
    gref = oracle.backward(*oracle_args(x, w), go, lse=ref["lse"], magnitudes=True,
                           **oracle_opts(w))
    check_backward(out, gref, tol, x["bias"] is not None, grad_kappas(w))


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_parity(w):
    _check_case(w)


def test_parity_mid_workload():
    """The bf16 mid workload exactly as specified: N=4096, H=2048, V=32000,
    bias, Zipf targets, 10% ignored, mean; full tensors compared."""
    _check_case(WORKLOADS["mid_bf16"])


@pytest.mark.parametrize("chunk", [256, 1024, 2304])
def test_parity_multi_chunk_backward(chunk):
    """The backward in several vocabulary chunks (the last one ragged), with a
    bias so grad_bias partials cross chunk boundaries."""
    w = _case("chunked", 520, 200, 5000, bias_var=0.02, softcap=20.0, ignore_frac=0.1)
    _check_case(w, vocab_chunk=chunk)


@pytest.mark.parametrize("dtype,skip", [("bf16", False), ("bf16", True), ("f16", False)])
def test_parity_narrow_last_chunk(dtype, skip):
    """V = 868 in vocabulary chunks of 256: the last chunk is 100 columns wide. At
    H <= 2048 the dlogits GEMM runs two epilogue warps per TMEM lane quarter, one
    per 128-column half of a tile; in the last chunk the second-half warps get no
    column but still take part in the grad_bias flush and the tile barriers."""
    w = _case("narrow_last_chunk", 700, 192, 868, dtype=dtype, bias_var=0.02, softcap=15.0,
              ignore_frac=0.1)
    _check_case(w, vocab_chunk=256, skip_ignored=skip)


@pytest.mark.parametrize("dtype,skip", [("bf16", True), ("f16", False)])
def test_parity_relay_narrow_last_chunk(dtype, skip):
    """H = 2112 > 2048: the forward and dlogits GEMMs run 4 epilogue warps with
    lane quarters 0 and 1 relayed through shared memory. V = 868 in chunks of
    256 leaves a 100-column last chunk, whose relayed chunks past the chunk's
    width are skipped, not read; a bias sends grad_bias partials through the
    relayed warps too."""
    w = _case("relay_narrow_last_chunk", 300, 2112, 868, dtype=dtype, bias_var=0.02,
              softcap=15.0, ignore_frac=0.1)
    _check_case(w, vocab_chunk=256, skip_ignored=skip)


@pytest.mark.parametrize("h", [37, 64])
def test_parity_f32_multi_chunk(h):
    """fp32 backward in six vocabulary chunks of 256, the last 219 wide (not a
    multiple of 4), with a bias: H = 37 runs the element-wise loads, H = 64 the
    16-byte ones with a ragged k tail in the grad_hidden contraction; N = 300
    leaves a 44-row tail in the third 128-row tile."""
    w = _case(f"f32_chunked_h{h}", 300, h, 1499, dtype="f32", bias_var=0.02, softcap=20.0,
              ignore_frac=0.1)
    _check_case(w, vocab_chunk=256)


def _misaligned(t):
    """A copy of `t` whose data starts 4 bytes past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 4, dtype=t.dtype, device=t.device)
    view = buf[1:1 + t.numel()].view(t.shape)
    view.copy_(t)
    assert view.data_ptr() % 16 == 4
    return view


def test_parity_f32_misaligned_inputs():
    """fp32 accepts any 4-byte-aligned hidden and weight: with both 4 bytes
    off a 16-byte boundary (H = 64 would otherwise take the vector loads) the
    kernels fall back to element-wise loads and give the same results."""
    w = _case("f32_misaligned", 200, 64, 900, dtype="f32", bias_var=0.02, ignore_frac=0.1)
    x = make_inputs(w)
    xd = to_dev(x)
    xd["hidden"] = _misaligned(xd["hidden"])
    xd["weight"] = _misaligned(xd["weight"])
    out = run_gpu(xd, w, grad_out=0.75)
    assert out["err_word"] == 0
    ref = oracle.forward(*oracle_args(x, w), **oracle_opts(w))
    tol = TOL[w.dtype]
    check_forward(out, ref, w, tol)
    gref = oracle.backward(*oracle_args(x, w), 0.75, lse=ref["lse"], magnitudes=True,
                           **oracle_opts(w))
    check_backward(out, gref, tol, True, grad_kappas(w))


def test_parity_grad_weight_fp32():
    """grad_weight kept in fp32 (accumulated in fp32 tensor memory, stored once)."""
    w = _case("gw_f32", 384, 256, 3000, ignore_frac=0.05)
    _check_case(w, grad_weight_dtype=torch.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_all_rows_ignored(dtype):
    """n_valid = 0: 'mean' loss and metrics are NaN, every gradient is 0."""
    w = _case("all_ignored", 200, 64, 700, dtype=dtype, bias_var=0.02, ignore_frac=1.0)
    x = make_inputs(w)
    out = run_gpu(to_dev(x), w)
    assert int(out["n_valid"]) == 0
    assert math.isnan(float(out["loss"]))
    assert math.isnan(float(out["metrics"][0])) and math.isnan(float(out["metrics"][1]))
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        assert torch.count_nonzero(out[k]) == 0, k


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_single_row_and_vocab_of_one(dtype):
    w = _case("one_row", 1, 64, 333, dtype=dtype, reduction="sum")
    _check_case(w)
    w1 = _case("v1", 50, 64, 1, dtype=dtype, reduction="mean", bias_var=0.02)
    x = make_inputs(w1)
    out = run_gpu(to_dev(x), w1)
    assert float(out["loss"]) == 0.0
    assert torch.all(out["lse_rows"] == out["lse_rows"])  # finite, no NaN
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        assert float(out[k].abs().max()) < 1e-6


@pytest.mark.parametrize("dtype,skip", [("bf16", False), ("bf16", True), ("f16", False),
                                        ("f32", False)])
def test_zero_weight_uniform_softmax(dtype, skip):
    """weight = 0 and bias = 0 make every logit 0, so the softmax is uniform:
    lse = loss = entropy = ln V on every valid row; all V logits tie, so the
    argmax is index 0 on every row (the lowest index wins across tiles and
    vocabulary splits); D = g (1/V - onehot), hence grad_hidden = D W = 0
    exactly and grad_bias_j = g (n_valid / V - #{valid rows with target j}).
    V = 5000 spans 20 vocabulary tiles with a ragged last one."""
    w = _case("zero_weight", 300, 64, 5000, dtype=dtype, bias_var=0.02, ignore_frac=0.1)
    x = make_inputs(w)
    x["weight"] = torch.zeros_like(x["weight"])
    x["bias"] = torch.zeros_like(x["bias"])
    t = x["targets"]
    valid = t != w.ignore_index
    t[((torch.arange(w.n) % 7) == 0) & valid] = 0  # some rows whose target is the argmax
    go = 0.75
    out = run_gpu(to_dev(x), w, grad_out=go, skip_ignored=skip)
    assert out["err_word"] == 0
    nv = int(valid.sum())
    lnv = math.log(w.v)
    assert int(out["n_valid"]) == nv
    lse = out["lse_rows"].double()[valid]
    assert torch.allclose(lse, torch.full_like(lse, lnv), rtol=1e-5, atol=0)
    expect_loss = torch.where(valid, torch.tensor(lnv, dtype=torch.float64), 0.0)
    assert torch.allclose(out["loss_rows"].double(), expect_loss, rtol=1e-5, atol=0)
    assert abs(float(out["loss"]) - lnv) <= 1e-5 * lnv
    hits = t[valid] == 0
    assert torch.equal(out["correct_rows"][valid] != 0, hits)
    assert abs(float(out["metrics"][0]) - float(hits.sum()) / nv) <= 1e-6
    ent = out["entropy_rows"].double()[valid]
    assert torch.allclose(ent, torch.full_like(ent, lnv), rtol=1e-4, atol=0)
    assert abs(float(out["metrics"][1]) - lnv) <= 1e-4 * lnv
    assert torch.count_nonzero(out["grad_hidden"]) == 0
    g = go / nv
    counts = torch.bincount(t[valid], minlength=w.v).double()
    expect_gb = g * (nv / w.v - counts)
    tol = TOL[w.dtype]
    ref = oracle.forward(*oracle_args(x, w), **oracle_opts(w))
    gref = oracle.backward(*oracle_args(x, w), go, lse=ref["lse"], magnitudes=True,
                           **oracle_opts(w))
    kap = grad_kappas(w)
    assert_grad_close("grad_bias (closed form)", out["grad_bias"], expect_gb, tol,
                      gref["grad_bias_mag"], kap["grad_bias"])
    check_backward(out, gref, tol, True, kap)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_empty_batch(dtype):
    """N = 0: 'sum' gives 0, 'mean' NaN, grad_weight and grad_bias are 0."""
    for red in ("sum", "mean"):
        w = _case("empty", 0, 64, 300, dtype=dtype, bias_var=0.02, reduction=red)
        x = make_inputs(w)
        out = run_gpu(to_dev(x), w)
        assert int(out["n_valid"]) == 0
        if red == "sum":
            assert float(out["loss"]) == 0.0
        else:
            assert math.isnan(float(out["loss"]))
        assert out["grad_hidden"].shape == (0, 64)
        assert torch.count_nonzero(out["grad_weight"]) == 0
        assert torch.count_nonzero(out["grad_bias"]) == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_target_out_of_range(dtype):
    """A target outside [0, V) that is not ignore_index sets the error word,
    gives that row a NaN loss and no gradient; other rows are unaffected."""
    w = _case("bad_target", 130, 64, 500, dtype=dtype, reduction="sum")
    x = make_inputs(w)
    x["targets"][5] = 500
    x["targets"][77] = -3
    out = run_gpu(to_dev(x), w)
    assert out["err_word"] & 1
    assert math.isnan(float(out["loss_rows"][5])) and math.isnan(float(out["loss_rows"][77]))
    assert math.isnan(float(out["loss"]))
    ref = oracle.forward(*oracle_args(x, w))
    ok = torch.ones(130, dtype=torch.bool)
    ok[[5, 77]] = False
    tol = TOL[dtype]
    assert_rows_close("loss_rows", out["loss_rows"], ref["loss"], tol["loss_rel"], ok,
                      floor=row_floor(w.h, ce_row_ops(ref)))
    gref = oracle.backward(*oracle_args(x, w), 1.0, lse=ref["lse"], magnitudes=True)
    check_backward(out, gref, tol, False, grad_kappas(w))


SKIP_CASES = [
    _case("skip_tails_cap_sum", 300, 136, 1000, bias_var=0.02, softcap=30.0, logit_scale=0.5,
          hidden_var=2.0, ignore_frac=0.3, reduction="sum"),
    _case("skip_none_4097", 4097, 512, 4096, ignore_frac=0.1, reduction="none"),
    _case("skip_zipf_bias", 640, 192, 5000, bias_var=0.02, targets="zipf", ignore_frac=0.45),
    _case("skip_most_ignored", 900, 256, 3000, ignore_frac=0.97, bias_var=0.02),
    _case("skip_none_ignored", 520, 128, 2000, ignore_frac=0.0),
]


@pytest.mark.parametrize("w", SKIP_CASES, ids=[w.name for w in SKIP_CASES])
def test_parity_skip_ignored(w):
    """Ignored rows left out of every contraction (FLCE_SKIP_IGNORED_ROWS):
    same loss, metrics and gradients as the oracle; the kept rows' lse."""
    _check_case(w, skip_ignored=True)


def test_parity_skip_ignored_multi_chunk():
    w = _case("skip_chunked", 777, 200, 5000, bias_var=0.02, softcap=20.0, ignore_frac=0.3)
    _check_case(w, vocab_chunk=1024, skip_ignored=True)


def test_skip_ignored_all_rows_ignored():
    w = _case("skip_all_ignored", 300, 64, 700, bias_var=0.02, ignore_frac=1.0)
    x = make_inputs(w)
    out = run_gpu(to_dev(x), w, skip_ignored=True)
    assert int(out["n_valid"]) == 0
    assert math.isnan(float(out["loss"]))
    assert torch.all(out["loss_rows"] == 0)
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        assert torch.count_nonzero(out[k]) == 0, k


F16_CASES = [
    _case("f16_tails_cap_sum", 300, 136, 1000, dtype="f16", bias_var=0.02, softcap=30.0,
          logit_scale=0.5, hidden_var=2.0, ignore_frac=0.3, reduction="sum"),
    _case("f16_mean_v32003", 512, 256, 32003, dtype="f16", ignore_frac=0.05),
    _case("f16_none", 700, 264, 3333, dtype="f16", bias_var=0.02, ignore_frac=0.1,
          reduction="none"),
    _case("f16_peaked_mean", 1024, 512, 8192, dtype="f16", peaked_frac=0.01, ignore_frac=0.05),
]


@pytest.mark.parametrize("w", F16_CASES, ids=[w.name for w in F16_CASES])
def test_parity_f16(w):
    """fp16 inputs on the tensor cores (the kernel card's signature lists
    float16); D is stored in fp16 times a power-of-two scale."""
    _check_case(w)


def test_parity_f16_skip_ignored_chunks():
    w = _case("f16_skip_chunks", 900, 200, 5000, dtype="f16", bias_var=0.02, softcap=20.0,
              ignore_frac=0.3)
    _check_case(w, vocab_chunk=1024, skip_ignored=True)


def test_f16_mean_workload_shape():
    """The mid workload's shape and recipe with fp16 inputs (N=4096, H=2048,
    V=32000, bias, Zipf targets, 10% ignored, mean)."""
    _check_case(WORKLOADS["mid_bf16"].with_shape(dtype="f16"))


OPT_CASES = [
    _case("ls_bf16_mean", 520, 256, 5000, bias_var=0.02, ignore_frac=0.1, label_smoothing=0.1),
    _case("zl_bf16_sum_cap", 300, 136, 1000, softcap=30.0, logit_scale=0.5, hidden_var=2.0,
          ignore_frac=0.3, reduction="sum", z_loss=1e-3),
    _case("ls_zl_bf16_none", 700, 264, 3333, bias_var=0.02, ignore_frac=0.1, reduction="none",
          label_smoothing=0.2, z_loss=1e-4),
    _case("ls_zl_f16_peaked", 1024, 512, 8192, dtype="f16", peaked_frac=0.01, ignore_frac=0.05,
          label_smoothing=0.05, z_loss=1e-3),
    _case("ls_zl_f32", 257, 96, 2100, dtype="f32", bias_var=0.5, reduction="sum",
          label_smoothing=0.1, z_loss=1e-3),
    # H > 2048: the relayed 4-warp epilogues carry the per-tile logit sums and the smoothed,
    # z-loss D for lane quarters 0 and 1
    _case("ls_zl_relay_h2112", 300, 2112, 1000, bias_var=0.02, softcap=15.0, ignore_frac=0.1,
          label_smoothing=0.1, z_loss=1e-3, return_metrics=True),
]


@pytest.mark.parametrize("w", OPT_CASES, ids=[w.name for w in OPT_CASES])
def test_parity_label_smoothing_zloss(w):
    """Label smoothing and z-loss (the CuTe-DSL FLCE pull request's options)."""
    _check_case(w)


def test_parity_label_smoothing_zloss_skip_chunks():
    w = _case("ls_zl_skip_chunks", 777, 200, 5000, bias_var=0.02, softcap=20.0, ignore_frac=0.3,
              label_smoothing=0.1, z_loss=1e-3)
    _check_case(w, vocab_chunk=1024, skip_ignored=True)
