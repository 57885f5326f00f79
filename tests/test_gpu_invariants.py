"""GPU invariants that hold at any size:
  * repeated forward and backward passes are bitwise identical;
  * return_metrics leaves the loss and the gradients bit-identical
    ("fused-linear-ce" model card, §Metrics for free);
  * the per-row loss does not depend on the backward's vocabulary chunking,
    and the gradients differ across chunkings only by fp32 summation order
    (the KL-divergence PR's partition-invariance note);
  * with softcap off and logit_scale 1, sum_j grad_bias_j = 0 (each row's
    p - onehot sums to zero over the vocabulary);
  * the autograd entry point returns the same gradients as the raw calls.
"""
import pytest
import torch

from _parity import run_gpu, to_dev
from linear_cross_entropy_vocab_gb300 import fused_linear_cross_entropy
from linear_cross_entropy_vocab_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _w(dtype="bf16", **kw):
    base = dict(bias_var=0.02, ignore_frac=0.1, softcap=20.0, logit_scale=0.8)
    base.update(kw)
    return Workload("inv", 700, 264, 3333, dtype, **base)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bitwise_repeatable(dtype):
    w = _w(dtype)
    xd = to_dev(make_inputs(w))
    a = run_gpu(xd, w)
    b = run_gpu(xd, w)
    for k in ("loss", "loss_rows", "lse_rows", "metrics", "correct_rows", "entropy_rows",
              "grad_hidden", "grad_weight", "grad_bias"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_metrics_leave_loss_and_grads_bit_identical(dtype):
    w = _w(dtype)
    x = to_dev(make_inputs(w))
    res = []
    for metrics in (False, True):
        h = x["hidden"].clone().requires_grad_(True)
        wt = x["weight"].clone().requires_grad_(True)
        b = x["bias"].clone().requires_grad_(True)
        out = fused_linear_cross_entropy(h, wt, x["targets"], b, softcap=w.softcap,
                                         logit_scale=w.logit_scale, return_metrics=metrics)
        loss = out[0] if metrics else out
        loss.backward()
        res.append((loss.detach().clone(), h.grad.clone(), wt.grad.clone(), b.grad.clone()))
        if metrics:
            m = out[1]
            assert set(m) == {"mean_token_accuracy", "entropy"}
            assert not m["entropy"].requires_grad
    for u, v in zip(res[0], res[1]):
        assert torch.equal(u, v)


@pytest.mark.parametrize("vocab_chunk", [0, 512])
def test_autograd_matches_raw_calls(vocab_chunk):
    """The autograd entry point leaves ignored rows out of the GEMMs; it equals
    the raw calls made with the same flag, and passes its vocab_chunk to the
    backward (512: seven chunks, bitwise the raw calls with that chunk)."""
    w = _w("bf16", reduction="sum")
    x = to_dev(make_inputs(w))
    raw = run_gpu(x, w, grad_out=1.0, skip_ignored=True, vocab_chunk=vocab_chunk)
    h = x["hidden"].clone().requires_grad_(True)
    wt = x["weight"].clone().requires_grad_(True)
    b = x["bias"].clone().requires_grad_(True)
    loss = fused_linear_cross_entropy(h, wt, x["targets"], b, softcap=w.softcap,
                                      logit_scale=w.logit_scale, reduction="sum",
                                      vocab_chunk=vocab_chunk)
    loss.backward()
    assert torch.equal(loss.detach().cpu(), raw["loss"])
    assert torch.equal(h.grad.cpu(), raw["grad_hidden"])
    assert torch.equal(wt.grad.cpu(), raw["grad_weight"])
    assert torch.equal(b.grad.cpu(), raw["grad_bias"])


# fp32 inputs: H = 262 runs the FFMA kernels (rows not a multiple of 16 bytes),
# H = 264 the tensor cores with operands split into three bf16 parts.
@pytest.mark.parametrize("dtype,h,bar", [("bf16", 264, 1e-2), ("f32", 262, 1e-5),
                                         ("f32", 264, 1e-4)],
                         ids=["bf16", "f32_ffma", "f32_split"])
def test_vocab_chunk_invariance(dtype, h, bar):
    """grad_hidden sums the chunks' products in fp32, so it depends on the
    chunking through the summation order only. bf16: D's rounding dominates
    (the bf16 normwise bar). FFMA: one fp32 rounding per product. Split
    operands: the tensor cores add each 16-term partial product into the fp32
    accumulator with their own rounding, so the order moves the sum by more;
    each chunking meets the fp32 normwise parity bar (1e-4) against the fp64
    oracle, and this bounds their difference by the same."""
    w = Workload("inv", 700, h, 3333, dtype, bias_var=0.02, ignore_frac=0.1, softcap=20.0,
                 logit_scale=0.8)
    x = to_dev(make_inputs(w))
    one = run_gpu(x, w, vocab_chunk=4096)  # a single chunk
    many = run_gpu(x, w, vocab_chunk=512)  # seven chunks
    assert torch.equal(one["loss_rows"], many["loss_rows"])
    # grad_weight and grad_bias rows come from the same tiles in both plans
    assert torch.equal(one["grad_weight"], many["grad_weight"])
    assert torch.equal(one["grad_bias"], many["grad_bias"])
    d = (one["grad_hidden"].double() - many["grad_hidden"].double()).norm()
    ref = one["grad_hidden"].double().norm()
    assert float(d / ref) < bar


def test_posterior_mass_identity():
    w = _w("f32", softcap=None, logit_scale=1.0, reduction="sum")
    x = to_dev(make_inputs(w))
    out = run_gpu(x, w)
    gb = out["grad_bias"].double()
    assert abs(float(gb.sum())) <= 1e-5 * float(gb.abs().sum())


@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_skip_ignored_matches_all_rows(reduction):
    """Leaving ignored rows out changes no kept row's result: loss rows, the
    kept rows' lse and grad_hidden are bitwise identical (each row's logits
    and gradient row do not depend on other rows); grad_weight and grad_bias
    sum the same terms in another order."""
    w = _w("bf16", reduction=reduction, ignore_frac=0.3)
    x = to_dev(make_inputs(w))
    go = torch.linspace(0.5, 1.5, w.n) if reduction == "none" else 1.0
    a = run_gpu(x, w, grad_out=go)
    b = run_gpu(x, w, grad_out=go, skip_ignored=True)
    keep = x["targets"].cpu() != w.ignore_index
    assert torch.equal(a["loss_rows"], b["loss_rows"])
    assert torch.equal(a["lse_rows"][keep], b["lse_rows"][keep])
    assert torch.equal(a["correct_rows"], b["correct_rows"])
    assert torch.equal(a["metrics"], b["metrics"])
    assert torch.equal(a["grad_hidden"], b["grad_hidden"])
    for k in ("grad_weight", "grad_bias"):
        d = (a[k].double() - b[k].double()).norm() / a[k].double().norm()
        assert float(d) < 1e-2, (k, float(d))


def test_leading_batch_dimensions_match_flattened_rows():
    """hidden [B, T, H] with targets [B, T] (and teacher probabilities
    [B, T, V] for KL) give bitwise the results of the flattened rows; 'none'
    returns per-position losses in the batch shape."""
    from linear_cross_entropy_vocab_gb300 import fused_linear_kl_div
    from linear_cross_entropy_vocab_gb300.workloads import make_teacher_probs

    w = Workload("batched", 600, 128, 1000, "bf16", ignore_frac=0.1)
    x = to_dev(make_inputs(w))
    q = make_teacher_probs(w).cuda()
    for reduction in ("mean", "none"):
        outs = []
        for shaped in (False, True):
            h = x["hidden"].clone().requires_grad_(True)
            wt = x["weight"].clone().requires_grad_(True)
            hin = h.reshape(2, 300, 128) if shaped else h
            tin = x["targets"].reshape(2, 300) if shaped else x["targets"]
            loss = fused_linear_cross_entropy(hin, wt, tin, reduction=reduction)
            if shaped and reduction == "none":
                assert loss.shape == (2, 300)
            loss.sum().backward()
            outs.append((loss.detach().reshape(-1).cpu(), h.grad.cpu(), wt.grad.cpu()))
        for u, v in zip(*outs):
            assert torch.equal(u, v)
    outs = []
    for shaped in (False, True):
        h = x["hidden"].clone().requires_grad_(True)
        hin = h.reshape(2, 300, 128) if shaped else h
        qin = q.reshape(2, 300, 1000) if shaped else q
        lab = x["targets"].reshape(2, 300) if shaped else x["targets"]
        loss = fused_linear_kl_div(hin, x["weight"], qin, lab, reduction="none")
        loss.sum().backward()
        outs.append((loss.detach().reshape(-1).cpu(), h.grad.cpu()))
    for u, v in zip(*outs):
        assert torch.equal(u, v)


def test_two_threads_two_streams_match_sequential():
    """Two host threads, each on its own CUDA stream, run forward+backward of
    different problems (bf16 cross-entropy with bias and softcap; fp16 KL
    divergence) at the same time. Per-thread library state (the error text,
    the tensor-map element type) and the kernels' independence from other
    grids must give bitwise the results of running them one after the
    other."""
    import threading

    from linear_cross_entropy_vocab_gb300 import fused_linear_kl_div
    from linear_cross_entropy_vocab_gb300.workloads import make_teacher_probs

    w1 = _w("bf16")
    x1 = to_dev(make_inputs(w1))
    w2 = Workload("thr_kl", 500, 256, 3000, "f16", ignore_frac=0.2)
    x2 = to_dev(make_inputs(w2))
    q2 = make_teacher_probs(w2).cuda()

    def job1():
        h = x1["hidden"].clone().requires_grad_(True)
        wt = x1["weight"].clone().requires_grad_(True)
        loss = fused_linear_cross_entropy(h, wt, x1["targets"], x1["bias"], softcap=w1.softcap,
                                          logit_scale=w1.logit_scale)
        loss.backward()
        return loss.detach(), h.grad, wt.grad

    def job2():
        h = x2["hidden"].clone().requires_grad_(True)
        wt = x2["weight"].clone().requires_grad_(True)
        loss = fused_linear_kl_div(h, wt, q2, x2["targets"], temperature=1.7)
        loss.backward()
        return loss.detach(), h.grad, wt.grad

    seq = [job1(), job2()]
    torch.cuda.synchronize()
    res, errs = [None, None], []

    def run(i, fn):
        try:
            with torch.cuda.stream(torch.cuda.Stream()):
                out = fn()
                torch.cuda.current_stream().synchronize()
            res[i] = out
        except Exception as e:  # reported below
            errs.append(e)

    ts = [threading.Thread(target=run, args=(0, job1)), threading.Thread(target=run, args=(1, job2))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    for a, b in zip(seq, res):
        for u, v in zip(a, b):
            assert torch.equal(u.cpu(), v.cpu())
