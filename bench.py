#!/usr/bin/env python3
"""Fused linear cross-entropy forward+backward throughput on GB300.

One step = flce_forward + flce_backward (all three gradients) over one batch of
the Llama-3 LM-head workload: N=8192 tokens, H=4096, V=128256, bf16, no bias,
2% ignored targets, reduction mean, metrics on. Inputs are seeded synthetic
tensors resident in HBM; the 1.05 GB weight exceeds the 129 MB L2, so no L2
flush is needed between steps.

Prints one JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle
instead, on a bounded sample of the same workload, on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from linear_cross_entropy_vocab_gb300.workloads import (  # noqa: E402
    WORKLOADS, gemm_flops, make_inputs, make_teacher_probs)

METRIC = "FLCE fwd+bwd tokens/s at H4096 V128256 bf16; % of dense-BF16 tensor peak"
KL_METRIC = "fused linear KL fwd+bwd tokens/s at H4096 V128256 bf16; % of dense-BF16 tensor peak"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "llama3_head_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# contractions of N x H x V per step of each tensor-core role: bwd_grads runs
# both gradient GEMMs (grad_hidden and grad_weight) in one launch per chunk
GEMM_ROLES = {"fwd_stats": 1, "fwd_kl": 1, "bwd_dlogits": 1, "bwd_dlogits_kl": 1,
              "bwd_grads": 2, "fwd_stats_split": 1, "bwd_dlogits_split": 1, "bwd_grads_split": 2,
              "fwd_kl_split": 1, "bwd_dlogits_kl_split": 1}
# fp32 inputs whose rows are a multiple of 16 bytes run on the tensor cores with
# each operand split into three bf16 parts: six bf16 products per fp32 product,
# so their peak is the bf16 peak / 6
SPLIT_ROLES = ("fwd_stats_split", "bwd_dlogits_split", "bwd_grads_split", "fwd_kl_split",
               "bwd_dlogits_kl_split")
SPLIT_PASSES = 6

# the fp32 path's contractions run on the FP32 FMA units (ALU-bound)
ALU_ROLES = ("fwd_stats_f32", "fwd_kl_f32", "bwd_dlogits_f32", "bwd_grad_weight_f32",
             "bwd_grad_hidden_f32")
FP32_LANES_PER_SM = 128  # FP32 FMA lanes per SM (4 schedulers x 32)


def strip_c_comments(src: str) -> str:
    """C/C++ source without its comments, whitespace runs collapsed to one
    space: what the compiler sees, so that editing a comment does not count
    as changing a kernel. String and character literals are kept verbatim."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sources_sha256() -> str:
    """Hash of the CUDA sources and the C header (comments stripped), in a
    fixed file order."""
    import glob
    import hashlib

    files = sorted(glob.glob(os.path.join(ROOT, "linear_cross_entropy_vocab_gb300", "csrc", "*")))
    files.append(os.path.join(ROOT, "include", "flce.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.relpath(f, ROOT).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(strip_c_comments(fh.read()).encode())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu capture, or
    None when the capture was taken on other kernel sources or workload."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        d = json.load(fh)
    if d.get("csrc_sha256") != kernel_sources_sha256():
        return None
    return d.get("workloads", {}).get(workload, {}).get("bytes_per_launch", {}).get(kernel)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_of(args):
    """The workload, with the --dtype / --forward-only variants applied."""
    w = WORKLOADS[args.workload]
    if args.dtype is not None:
        w = w.with_shape(dtype=args.dtype)
    if args.forward_only and w.name == "long_bf16":
        w = w.with_shape(reduction="none")  # this workload's forward-only phase
    if args.label_smoothing or args.z_loss:
        w = w.with_shape(label_smoothing=args.label_smoothing, z_loss=args.z_loss)
    return w


def describe(w) -> str:
    parts = [f"{w.name}: N={w.n} H={w.h} V={w.v} {w.dtype}",
             "bias" if w.bias_var is not None else "no bias",
             f"{round(100 * w.ignore_frac)}% ignore_index", f"{w.targets} targets"]
    if w.softcap:
        parts.append(f"logit_scale={w.logit_scale} softcap={w.softcap}")
    if w.peaked_frac:
        parts.append(f"{round(100 * w.peaked_frac)}% weight rows x{w.peaked_factor:g}")
    if w.label_smoothing or w.z_loss:
        parts.append(f"label_smoothing={w.label_smoothing:g} z_loss={w.z_loss:g}")
    parts.append(w.reduction + (", return_metrics" if w.return_metrics else ""))
    return ", ".join(parts)


# KL divergence workload: the Llama-3 head shape that the KL pull request
# benchmarks (8192 x 4096 x 128256, bf16), teacher probabilities from
# make_teacher_probs, the workload's targets as labels (2% ignored, left out
# of the contractions), temperature 1, batchmean.
KL_TEMPERATURE = 1.0
KL_REDUCTION = "batchmean"


def describe_kl(w) -> str:
    return (f"fused linear KL, {w.name} shape: N={w.n} H={w.h} V={w.v} {w.dtype}, "
            f"{'bias' if w.bias_var is not None else 'no bias'}, teacher = softmax of "
            f"N(0, 4) logits, labels with {round(100 * w.ignore_frac)}% ignore_index, "
            f"T={KL_TEMPERATURE:g}, {KL_REDUCTION}")


def make_bench_inputs(w, kl: bool) -> dict:
    x = make_inputs(w)
    if kl:
        x["q"] = make_teacher_probs(w)
    return x


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.path = tempfile.mktemp(prefix="flce_clocks_", suffix=".csv")
        self.proc = None
        self.device_id = device_id

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", self.device_id],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- ranks
def max_over_ranks(value: float, world: int, device) -> float:
    """The largest `value` over the ranks of the default process group (the
    slowest rank's time); `value` itself on one rank. `device` is where the
    reduction runs: the GPU for NCCL, the CPU for gloo."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput of `world` replicas that each processed
    `tokens_per_rank` tokens per step for `steps` steps, timed by the slowest
    rank (weak scaling: the work per GPU is fixed)."""
    return world * tokens_per_rank * steps / (max_ms / 1e3)


# ----------------------------------------------------------------- our arm
class Step:
    """Preallocated buffers and the two C-ABI calls of one fwd+bwd step."""

    def __init__(self, x: dict, w, dev, skip_ignored: bool = True, forward_only: bool = False,
                 vocab_chunk: int = 0):
        from linear_cross_entropy_vocab_gb300 import abi

        self.abi = abi
        self.x = x
        self.w = w
        self.forward_only = forward_only
        n, h = x["hidden"].shape
        v = x["weight"].shape[0]
        code = {torch.bfloat16: abi.FLCE_BF16, torch.float16: abi.FLCE_F16,
                torch.float32: abi.FLCE_F32}[x["hidden"].dtype]
        self.prob = abi.make_problem(n, h, v, code, x["bias"] is not None, w.ignore_index,
                                     w.logit_scale, w.softcap, w.reduction,
                                     vocab_chunk=vocab_chunk, skip_ignored=skip_ignored,
                                     label_smoothing=w.label_smoothing, z_loss=w.z_loss)
        f32 = dict(dtype=torch.float32, device=dev)
        self.loss_rows = torch.empty(n, **f32)
        self.lse_rows = torch.empty(n, **f32)
        self.loss = torch.empty((), **f32)
        self.metrics = torch.empty(2, **f32) if w.return_metrics else None
        self.n_valid = torch.empty((), dtype=torch.int32, device=dev)
        self.err = torch.zeros((), dtype=torch.int32, device=dev)
        self.grad_out = torch.ones((), **f32)
        self.gh = torch.empty_like(x["hidden"])
        self.gw = torch.empty_like(x["weight"])
        self.gb = None if x["bias"] is None else torch.empty_like(x["bias"])
        self.ws_f = abi.flce_forward_workspace_size(self.prob)
        self.ws_b = abi.flce_backward_workspace_size(self.prob)
        self.ws = torch.empty(max(self.ws_f, self.ws_b), dtype=torch.uint8, device=dev)

    def rebind(self, x: dict) -> "Step":
        """The same step (problem, outputs, workspace) on other input buffers."""
        other = object.__new__(type(self))
        other.__dict__.update(self.__dict__)
        other.x = x
        return other

    def __call__(self, stream):
        a, x, p = self.abi, self.x, lambda t: None if t is None else t.data_ptr()
        a.flce_forward(self.prob, p(x["hidden"]), p(x["weight"]), p(x["bias"]), p(x["targets"]),
                       p(self.loss_rows), p(self.lse_rows), None, None,
                       None if self.w.reduction == "none" else p(self.loss),
                       p(self.metrics), p(self.n_valid), p(self.err), p(self.ws), self.ws_f,
                       stream)
        if self.forward_only:
            return
        a.flce_backward(self.prob, p(x["hidden"]), p(x["weight"]), p(x["bias"]),
                        p(x["targets"]), p(self.lse_rows), p(self.n_valid), p(self.grad_out),
                        p(self.gh), p(self.gw), p(self.gb), p(self.err), p(self.ws), self.ws_b,
                        stream)


class KLStep:
    """Preallocated buffers and the two C-ABI calls of one fused linear KL
    fwd+bwd step."""

    def __init__(self, x: dict, w, dev, skip_ignored: bool = True, forward_only: bool = False,
                 vocab_chunk: int = 0):
        from linear_cross_entropy_vocab_gb300 import abi

        self.abi = abi
        self.x = x
        self.w = w
        self.forward_only = forward_only
        n, h = x["hidden"].shape
        v = x["weight"].shape[0]
        code = {torch.bfloat16: abi.FLCE_BF16, torch.float16: abi.FLCE_F16,
                torch.float32: abi.FLCE_F32}[x["hidden"].dtype]
        self.prob = abi.make_kl_problem(n, h, v, code, x["bias"] is not None, w.ignore_index,
                                        KL_TEMPERATURE, 1e-10, KL_REDUCTION,
                                        vocab_chunk=vocab_chunk, skip_ignored=skip_ignored)
        f32 = dict(dtype=torch.float32, device=dev)
        self.loss_rows = torch.empty(n, **f32)
        self.lse_rows = torch.empty(n, **f32)
        self.qsum_rows = torch.empty(n, **f32)
        self.loss = torch.empty((), **f32)
        self.metrics = None
        self.n_valid = torch.empty((), dtype=torch.int32, device=dev)
        self.err = torch.zeros((), dtype=torch.int32, device=dev)
        self.grad_out = torch.ones((), **f32)
        self.gh = torch.empty_like(x["hidden"])
        self.gw = torch.empty_like(x["weight"])
        self.gb = None if x["bias"] is None else torch.empty_like(x["bias"])
        self.ws_f = abi.flce_kl_forward_workspace_size(self.prob)
        self.ws_b = abi.flce_kl_backward_workspace_size(self.prob)
        self.ws = torch.empty(max(self.ws_f, self.ws_b), dtype=torch.uint8, device=dev)

    rebind = Step.rebind

    def __call__(self, stream):
        a, x, p = self.abi, self.x, lambda t: None if t is None else t.data_ptr()
        a.flce_kl_forward(self.prob, p(x["hidden"]), p(x["weight"]), p(x["bias"]), p(x["q"]),
                          p(x["targets"]), p(self.loss_rows), p(self.lse_rows),
                          p(self.qsum_rows), p(self.loss), p(self.n_valid), p(self.err),
                          p(self.ws), self.ws_f, stream)
        if self.forward_only:
            return
        a.flce_kl_backward(self.prob, p(x["hidden"]), p(x["weight"]), p(x["bias"]), p(x["q"]),
                           p(x["targets"]), p(self.lse_rows), p(self.qsum_rows),
                           p(self.n_valid), p(self.grad_out), p(self.gh), p(self.gw),
                           p(self.gb), p(self.err), p(self.ws), self.ws_b, stream)


def bench_ours(args, rank, world, dev):
    from linear_cross_entropy_vocab_gb300 import abi, api, native_build

    native_build.build()
    w = workload_of(args)
    xc = make_bench_inputs(w, args.kl)
    x = {k: (None if t is None else t.to(dev)) for k, t in xc.items()}
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    step = (KLStep if args.kl else Step)(x, w, dev, skip_ignored=not args.all_rows,
                                         forward_only=args.forward_only,
                                         vocab_chunk=args.vocab_chunk)
    n, h, v = w.n, w.h, w.v

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(max(args.warmup, 3)):
        step(sh)
    torch.cuda.synchronize(dev)
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error word {int(step.err.item())}")

    # ------------------------------------------------------ device-timed region
    clocks = ClockSampler(_smi_id(dev))
    clocks.start()
    barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(sh)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms = t0.elapsed_time(t1)
    clk = clocks.stop()
    ms = max_over_ranks(ms, world, dev)
    # per-kernel times: a second pass of the same steps with CUDA events
    # around every launch (events between launches keep the backward's
    # launches from overlapping, so they are not recorded in the timed region)
    abi.flce_profile_enable(True)
    torch.cuda.synchronize(dev)
    for _ in range(args.steps):
        step(sh)
    torch.cuda.synchronize(dev)
    prof, dropped = abi.flce_profile_collect()
    abi.flce_profile_enable(False)

    # ------------------------------------------------------ end to end (host buffers)
    # Every step copies its inputs from pinned host memory and reads its loss
    # (and metrics) back. Inputs are double-buffered: the copy of step i+1
    # runs on a side stream while step i computes. Measured twice: copying
    # every input each step (the weight too: the `e2e` figure), and copying
    # only the per-step activations -- hidden, targets and, for the KL
    # divergence, the teacher probabilities -- with the weight and bias
    # resident in HBM as a training loop keeps them.
    pin = {k: (None if t is None else t.pin_memory()) for k, t in xc.items()}
    loss_h = torch.empty((), dtype=torch.float32).pin_memory()
    met_h = torch.empty(2, dtype=torch.float32).pin_memory()
    # as many steps as the device-timed region, so that both run as long under
    # the power cap
    e2e_steps = max(2, args.steps)
    d2h = loss_h.numel() * 4 + (met_h.numel() * 4 if step.metrics is not None else 0)
    bufs = [x, {k: (None if t is None else t.clone()) for k, t in x.items()}]
    steps2 = [step, step.rebind(bufs[1])]
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_measure(keys):
        """ms for e2e_steps steps copying the inputs in `keys` every step,
        and the bytes copied per step."""
        def issue_copy(b):
            with torch.cuda.stream(copy_stream):
                for k in keys:
                    if pin[k] is not None:
                        bufs[b][k].copy_(pin[k], non_blocking=True)
                copied[b].record(copy_stream)

        def run(nsteps):
            issue_copy(0)
            for i in range(nsteps):
                b = i % 2
                if i + 1 < nsteps:
                    if i >= 1:
                        copy_stream.wait_event(done[1 - b])
                    issue_copy(1 - b)
                stream.wait_event(copied[b])
                steps2[b](sh)
                done[b].record(stream)
                loss_h.copy_(steps2[b].loss, non_blocking=True)
                if steps2[b].metrics is not None:
                    met_h.copy_(steps2[b].metrics, non_blocking=True)

        run(2)
        torch.cuda.synchronize(dev)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_event(e0)
        run(e2e_steps)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        nbytes = sum(pin[k].numel() * pin[k].element_size() for k in keys if pin[k] is not None)
        return max_over_ranks(e0.elapsed_time(e1), world, dev), nbytes

    # host link bandwidth: one copy of a step's inputs alone, on the copy stream
    all_keys = [k for k in pin if pin[k] is not None]
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    c0.record(copy_stream)
    with torch.cuda.stream(copy_stream):
        for k in all_keys:
            bufs[0][k].copy_(pin[k], non_blocking=True)
    c1.record(copy_stream)
    torch.cuda.synchronize(dev)
    h2d_all = sum(pin[k].numel() * pin[k].element_size() for k in all_keys)
    h2d_gbs = h2d_all / (c0.elapsed_time(c1) / 1e3) / 1e9

    e2e_ms, h2d = e2e_measure(all_keys)
    act_keys = [k for k in ("hidden", "targets", "q") if k in pin and pin[k] is not None]
    e2e_act_ms, h2d_act = e2e_measure(act_keys)
    del bufs, steps2

    # ------------------------------------------------------ peak memory of the public API
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    hh = x["hidden"].detach().requires_grad_(True)
    ww = x["weight"].detach().requires_grad_(True)
    if args.kl:
        loss = api.fused_linear_kl_div(hh, ww, x["q"], x["targets"],
                                       temperature=KL_TEMPERATURE, reduction=KL_REDUCTION,
                                       vocab_chunk=args.vocab_chunk)
    else:
        loss, _m = api.fused_linear_cross_entropy(hh, ww, x["targets"], return_metrics=True,
                                                  vocab_chunk=args.vocab_chunk)
    loss.backward()
    torch.cuda.synchronize(dev)
    peak_incr = torch.cuda.max_memory_allocated(dev) - base
    del hh, ww, loss

    peaks, peak_src = load_peaks()
    flops_step = gemm_flops(n, h, v) / (4.0 if args.forward_only else 1.0)
    tok_s = job_tokens_per_s(n, args.steps, world, ms)
    n_valid = int(step.n_valid.item())
    achieved_step = flops_step * args.steps / (ms / 1e3) / 1e12
    # dominant kernel: the role with the largest share of device time
    roles = {k: val for k, val in prof.items()}
    dom = max(roles, key=lambda k: roles[k][1]) if roles else None
    roofline = None
    if dom is not None:
        launches, tot_ms = roles[dom]
        # algorithmic work of one launch: the rows it computes (ignored rows
        # are left out of every contraction unless --all-rows; the fp32 path
        # computes every row)
        n_work = n if (args.all_rows or dom in ALU_ROLES or dom in SPLIT_ROLES) else n_valid
        roofline = roofline_entry(dom, launches, tot_ms, args.steps, n_work, h, v, ms, peaks,
                                  peak_src,
                                  torch.cuda.get_device_properties(dev).multi_processor_count)
        roofline["traffic"] = measured_traffic(dom, traffic_key(w, args))
        roofline["traffic_source"] = ("profiles/dram_traffic.json (ncu dram__bytes_read.sum + "
                                      "dram__bytes_write.sum per launch; null if the kernels "
                                      "changed since)")
    kernels = {k: {"launches": val[0], "ms_per_step": round(val[1] / args.steps, 4),
                   "share": round(val[1] / sum(u[1] for u in roles.values()), 4)}
               for k, val in roles.items()}
    kernels_how = ("a second pass of the timed steps with CUDA events around every "
                       "launch, on the launching stream; those events serialise launches that "
                       "overlap in the timed region, so the per-kernel sum can exceed "
                       "ms_per_step")
    out = {
        "metric": KL_METRIC if args.kl else METRIC,
        "value": round(tok_s, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic, seeded (distributions as in the workload description)",
        "config": {"workload": describe_kl(w) if args.kl else describe(w),
                   "global_batch": n * world, "seq_len": None,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": (f"inputs {input_bytes(x) / 2**20:.0f} MiB, L2 {L2_BYTES >> 20} MiB: "
                          "no flush between steps"),
                   "skip_ignored_rows": not args.all_rows,
                   "vocab_chunk": args.vocab_chunk or "library default",
                   "step": "forward only" if args.forward_only else "forward+backward"},
        "tensor_peak_frac": {
            "achieved_tflops": round(achieved_step, 1),
            "of_burst": round(achieved_step / peaks["bf16_tflops"], 4),
            "of_sustained": round(achieved_step / peaks["bf16_tflops_sustained"], 4),
            "of_burst_valid_rows": round(achieved_step * n_valid / n / peaks["bf16_tflops"], 4),
            "flops_per_step": flops_step, "peaks": peak_src,
            # fp32 operands split into bf16 parts: six bf16 products per fp32 product
            **({"of_split_burst": round(achieved_step / (peaks["bf16_tflops"] / SPLIT_PASSES), 4)}
               if any(r in SPLIT_ROLES for r in roles) else {})},
        "roofline": roofline,
        "kernels": kernels,
        "kernels_how": kernels_how,
        "gpu_launches": int(sum(val[0] for val in roles.values())),
        "gpu_launches_how": "launches of this library's kernels in the profiled pass of the "
                            "same steps (same launch sequence as the timed region)",
        "profile_dropped": dropped,
        "e2e": {"value": round(job_tokens_per_s(n, e2e_steps, world, e2e_ms), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "copies": "every input (weight included) pinned host -> device each step, on a "
                          "side stream, double-buffered",
                "h2d_gb_per_s": round(h2d_gbs, 1),
                "activations_only": {
                    "value": round(job_tokens_per_s(n, e2e_steps, world, e2e_act_ms), 1),
                    "unit": UNIT, "h2d_bytes_per_step": h2d_act, "d2h_bytes_per_step": d2h,
                    "copies": "+".join(act_keys) + " each step; weight and bias resident"}},
        "clocks": clk,
        "memory": {"peak_incremental_bytes_public_api": int(peak_incr),
                   "nxv_bf16_bytes": n * v * 2,
                   "workspace_fwd_bytes": step.ws_f, "workspace_bwd_bytes": step.ws_b},
    }
    return out


# ----------------------------------------------------------------- other workloads
# Every workload besides the headline one, measured in the same process after
# it: (key, workload name, options). The long batch is measured in both of its
# phases: forward only with reduction none, then forward+backward with mean.
PER_CONFIG = (
    ("tiny_fp32", "tiny_fp32", {}),
    # the oracle times all 4096 rows here (about 8 s on 16 cores), not a sample
    ("mid_bf16", "mid_bf16", {"cpu_budget_s": 14.0}),
    ("softcap_bf16", "softcap_bf16", {}),
    ("long_bf16_forward_none", "long_bf16", {"forward_only": True}),
    ("long_bf16", "long_bf16", {}),
    ("llama3_head_bf16_kl", "llama3_head_bf16", {"kl": True}),
)
L2_BYTES = 129 << 20
PER_CONFIG_TIMED_S = 0.4  # device time per workload's timed region (at least `steps` steps)


def input_bytes(x) -> int:
    """Bytes of a step's input tensors (a dict of tensors or None)."""
    return sum(t.numel() * t.element_size() for t in x.values() if t is not None)


def _flush_l2(buf):
    buf.add_(1)  # writes 2 x L2 of memory: nothing of the last step stays in L2


def measure_config(w, dev, steps, warmup, peaks, peak_src, forward_only=False, kl=False,
                   cpu_budget_s=6.0, with_cpu=True):
    """One workload: device-timed fwd(+bwd) steps through the C ABI (ignored
    rows left out of the contractions), the dominant kernel's share, the
    clock, peak incremental memory of one public-API step, and the oracle
    timed on a bounded sample of the workload's rows."""
    from linear_cross_entropy_vocab_gb300 import abi, api

    xc = make_bench_inputs(w, kl)
    x = {k: (None if t is None else t.to(dev)) for k, t in xc.items()}
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    step = (KLStep if kl else Step)(x, w, dev, skip_ignored=True, forward_only=forward_only)
    in_bytes = input_bytes(x)
    flush = None
    if in_bytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(max(warmup, 3)):
        step(sh)
    torch.cuda.synchronize(dev)
    # steps: enough for about PER_CONFIG_TIMED_S of device time
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    step(sh)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    est = max(t0.elapsed_time(t1), 1e-3)
    k = int(min(2000, max(steps, PER_CONFIG_TIMED_S * 1e3 / est)))
    clocks = ClockSampler(_smi_id(dev))
    clocks.start()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(k if flush is not None else 1)]
    if flush is not None:
        # per-step events, L2 written over between steps (inputs smaller than L2)
        for a, b in ev:
            _flush_l2(flush)
            a.record(stream)
            step(sh)
            b.record(stream)
    else:
        ev[0][0].record(stream)
        for _ in range(k):
            step(sh)
        ev[0][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in ev)
    clk = clocks.stop()
    abi.flce_profile_enable(True)  # per-kernel shares from a second, event-bracketed pass
    for _ in range(min(k, 50)):
        step(sh)
    torch.cuda.synchronize(dev)
    prof, _dropped = abi.flce_profile_collect()
    abi.flce_profile_enable(False)
    if int(step.err.item()) != 0:
        raise RuntimeError(f"{w.name}: device error word {int(step.err.item())}")
    n_valid = int(step.n_valid.item())
    del step
    # peak memory of one public-API step
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    hh = x["hidden"].detach().requires_grad_(not forward_only)
    ww = x["weight"].detach().requires_grad_(not forward_only)
    bb = None if x["bias"] is None else x["bias"].detach().requires_grad_(not forward_only)
    if kl:
        loss = api.fused_linear_kl_div(hh, ww, x["q"], x["targets"], bb,
                                       temperature=KL_TEMPERATURE, reduction=KL_REDUCTION)
    else:
        loss = api.fused_linear_cross_entropy(hh, ww, x["targets"], bb, w.ignore_index,
                                              w.logit_scale, w.softcap, w.reduction,
                                              return_metrics=w.return_metrics)
        if w.return_metrics:
            loss = loss[0]
    if not forward_only:
        (loss.sum() if loss.dim() else loss).backward()
    torch.cuda.synchronize(dev)
    peak_incr = torch.cuda.max_memory_allocated(dev) - base
    del hh, ww, bb, loss, flush
    n, h, v = w.n, w.h, w.v
    flops = gemm_flops(n, h, v) / (4.0 if forward_only else 1.0)
    t_step = ms / k / 1e3
    # fp32 inputs run split on the tensor cores or on the FFMA kernels (the
    # library decides by size); the launches profiled say which
    split = any(r in SPLIT_ROLES for r in (prof or {}))
    alu = w.dtype == "f32" and not split
    out = {
        "workload": describe_kl(w) if kl else describe(w),
        "step": "forward only" if forward_only else "forward+backward",
        "steps": k, "ms_per_step": round(ms / k, 4), "tokens_per_s": round(n / t_step, 1),
        "achieved_tflops": round(flops / t_step / 1e12, 2),
        "l2": ("L2 written over between steps (inputs smaller than L2)" if len(ev) > 1
               else f"inputs {in_bytes / 1e6:.0f} MB > L2, no flush"),
        "clocks": {"sm_mhz": clk.get("sm_mhz"), "reasons": clk.get("reasons"),
                   "samples": clk.get("samples")},
        "memory": {"peak_incremental_bytes_public_api": int(peak_incr),
                   "nxv_bytes": n * v * x["hidden"].element_size(),
                   "of_nxv": round(peak_incr / (n * v * x["hidden"].element_size()), 4),
                   "nxv": "one N x V logit matrix in the input type"},
    }
    if alu:
        mhz = peaks.get("sm_max_mhz", 2070.0)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        fma_peak = sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
        out["fp32_fma_peak_frac"] = round(flops / t_step / 1e12 / fma_peak, 4)
    elif split:
        a = flops / t_step / 1e12
        out["tensor_peak_frac"] = {
            "of_split_burst": round(a / (peaks["bf16_tflops"] / SPLIT_PASSES), 4),
            "split": f"fp32 operands as three bf16 parts: {SPLIT_PASSES} bf16 products per "
                     f"fp32 product, peak = bf16 burst / {SPLIT_PASSES}",
            "peaks": peak_src}
    else:
        a = flops / t_step / 1e12
        out["tensor_peak_frac"] = {
            "of_burst": round(a / peaks["bf16_tflops"], 4),
            "of_sustained": round(a / peaks["bf16_tflops_sustained"], 4),
            "of_burst_kept_rows": round(a * n_valid / n / peaks["bf16_tflops"], 4),
            "kept_rows": n_valid, "peaks": peak_src}
    if prof:
        dom = max(prof, key=lambda r: prof[r][1])
        out["dominant_kernel"] = {"kernel": dom, "share": round(
            prof[dom][1] / sum(u[1] for u in prof.values()), 4)}
    del x
    torch.cuda.empty_cache()
    if with_cpu:
        out["cpu_baseline"] = cpu_baseline(xc, w, budget_s=cpu_budget_s, kl=kl)
    return out


def _smi_id(dev) -> str:
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return str(torch.cuda.current_device())


def traffic_key(w, args) -> str:
    """Key of a workload variant in profiles/dram_traffic.json."""
    key = w.name + ("+kl" if args.kl else "") + ("+fwd" if args.forward_only else "")
    return key + ("+all_rows" if args.all_rows else "")


# ----------------------------------------------------------------- oracle timing
def _oracle_sample_step(xc, w, rows):
    import oracle

    sl = {k: (None if t is None else (t[:rows] if k in ("hidden", "targets") else t))
          for k, t in xc.items()}
    args = (sl["hidden"], sl["weight"], sl["targets"], sl["bias"], w.ignore_index,
            w.logit_scale, w.softcap, w.reduction)
    f = oracle.forward(*args)
    oracle.backward(*args, 1.0, lse=f["lse"])


def _oracle_kl_sample_step(xc, w, rows):
    from oracle import kl_oracle

    args = (xc["hidden"][:rows], xc["weight"], xc["q"][:rows], xc["bias"],
            xc["targets"][:rows], w.ignore_index, KL_TEMPERATURE, 1e-10, KL_REDUCTION)
    kl_oracle.forward(*args)
    kl_oracle.backward(*args, 1.0)


def _calibrate_rows(xc, w, budget_s, max_rows, kl=False):
    """Rows per sample so that one oracle step takes at most about budget_s
    (linear in the rows of a 64-row trial, fixed costs included)."""
    run = _oracle_kl_sample_step if kl else _oracle_sample_step
    t = time.perf_counter()
    run(xc, w, 64)
    per_row = (time.perf_counter() - t) / 64
    rows = int(budget_s / per_row)
    return max(8, min(max_rows, rows)), per_row


def cpu_model() -> str:
    """The host CPU's model name, as /proc/cpuinfo gives it (x86 and Arm)."""
    try:
        with open("/proc/cpuinfo") as fh:
            info = fh.read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "Hardware"):
        for line in info:
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    for line in info:  # Arm: implementer and part numbers only
        if line.startswith("CPU part") and ":" in line:
            return "Arm CPU part " + line.split(":", 1)[1].strip()
    return "unknown"


def cpu_baseline(xc, w, budget_s=15.0, kl=False):
    """The oracle's fp64 forward+backward on the first rows of the workload
    (all of them when they fit the budget), as tokens/s. A sample of fewer
    rows than the workload is extrapolated linearly in the rows: every row
    costs the same full-vocabulary work."""
    rows, _ = _calibrate_rows(xc, w, budget_s, w.n, kl)
    t = time.perf_counter()
    (_oracle_kl_sample_step if kl else _oracle_sample_step)(xc, w, rows)
    dt = time.perf_counter() - t
    what = "fused linear KL " if kl else ""
    full = rows >= w.n
    return {"value": round(rows / dt, 2), "unit": UNIT, "cores": torch.get_num_threads(),
            "cpu_model": cpu_model(), "kind": "oracle", "extrapolated": not full,
            "sample": (f"fp64 {what}forward+backward of all {rows} rows of the workload; "
                       f"{dt:.1f} s" if full else
                       f"fp64 {what}forward+backward of the first {rows} of {w.n} rows of the "
                       f"workload (full H={w.h}, V={w.v}) as one batch, {dt:.1f} s; "
                       f"tokens/s extrapolated linearly in the rows")}


def bench_reference(args):
    w = workload_of(args)
    xc = make_bench_inputs(w, args.kl)
    run = _oracle_kl_sample_step if args.kl else _oracle_sample_step
    total_budget = 150.0  # seconds for warmup + timed steps
    per_step = total_budget / (args.steps + max(args.warmup, 3))
    rows, _ = _calibrate_rows(xc, w, per_step, w.n, args.kl)
    for _ in range(max(args.warmup, 3)):
        run(xc, w, rows)
    t = time.perf_counter()
    for _ in range(args.steps):
        run(xc, w, rows)
    dt = time.perf_counter() - t
    val = round(rows * args.steps / dt, 2)
    what = "fused linear KL " if args.kl else ""
    sample = (f"each step: fp64 {what}forward+backward of the first {rows} rows of the "
              f"workload (full H={w.h}, V={w.v})")
    return {
        "impl": "reference", "metric": KL_METRIC if args.kl else METRIC, "value": val,
        "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe_kl(w) if args.kl else describe(w),
                   "global_batch": rows},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": torch.get_num_threads(),
                         "cpu_model": cpu_model(), "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }



def roofline_entry(dom, launches, tot_ms, steps, n_work, h, v, run_ms, peaks, peak_src, sms):
    """The `roofline` object of the dominant kernel `dom`, which ran `launches`
    times in `tot_ms` over `steps` timed steps of a `run_ms` timed region.

    achieved = the launch's algorithmic flops (2 n_work h v per step, split
    over its launches per step) / its average duration. A kernel timed inside
    a region of a second or more runs at the power-capped clock, so it is set
    against the sustained bf16 peak, a shorter one against the burst peak; the
    fp32 (FFMA) roles against sms x 128 FP32 lanes x 2 flops x the maximum SM
    clock."""
    alu = dom in ALU_ROLES
    per_step_flops = 2.0 * n_work * h * v * (GEMM_ROLES.get(dom, 0) or (1 if alu else 0))
    flops_per_launch = per_step_flops / (launches / steps)
    avg_ms = tot_ms / launches
    achieved = flops_per_launch / (avg_ms / 1e3) / 1e12
    if alu:
        mhz = peaks.get("sm_max_mhz", 2070.0)
        peak = round(sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12, 1)
        peak_kind = (f"fp32 FMA: {sms} SMs x {FP32_LANES_PER_SM} lanes x 2 FLOP x "
                     f"{mhz:g} MHz (unit counts and maximum clock)")
    else:
        long_run = run_ms >= 1000.0
        peak = peaks["bf16_tflops_sustained"] if long_run else peaks["bf16_tflops"]
        peak_kind = (f"bf16 {'sustained' if long_run else 'burst'}, {peak_src} "
                     f"(timed region {run_ms / 1e3:.2f} s)")
        if dom in SPLIT_ROLES:
            peak = round(peak / SPLIT_PASSES, 1)
            peak_kind += (f" / {SPLIT_PASSES}: fp32 operands as three bf16 parts, "
                          f"{SPLIT_PASSES} bf16 products per fp32 product")
    return {"bound": "alu" if alu else "tensor", "kernel": dom,
            "achieved": round(achieved, 1),
            "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "peak_kind": peak_kind,
            "flops_per_launch": flops_per_launch, "rows_per_launch": n_work,
            "avg_launch_ms": round(avg_ms, 4)}

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure the headline workload only (skip the per_config block)")
    ap.add_argument("--dtype", choices=["bf16", "f16", "f32"], default=None,
                    help="run the workload with this input type (default: the workload's)")
    ap.add_argument("--forward-only", action="store_true",
                    help="time flce_forward alone (the long workload uses reduction none)")
    ap.add_argument("--vocab-chunk", type=int, default=0,
                    help="vocabulary columns of the backward's dlogits buffer (0: the library's "
                         "default)")
    ap.add_argument("--label-smoothing", type=float, default=0.0)
    ap.add_argument("--z-loss", type=float, default=0.0)
    ap.add_argument("--all-rows", action="store_true",
                    help="run ignored rows through the GEMMs too (FLCE_SKIP_IGNORED_ROWS off)")
    ap.add_argument("--kl", action="store_true",
                    help="time the fused linear KL divergence (flce_kl_forward + "
                         "flce_kl_backward) on the workload's shape instead")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(bench_reference(args)), flush=True)
        return

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl", device_id=dev)
    out = bench_ours(args, rank, world, dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        w = workload_of(args)
        out["cpu_baseline"] = cpu_baseline(make_bench_inputs(w, args.kl), w, kl=args.kl)
    if not args.no_per_config and world == 1:
        peaks, peak_src = load_peaks()
        per = {}
        for key, name, opts in PER_CONFIG:
            wk = WORKLOADS[name]
            if opts.get("forward_only") and name == "long_bf16":
                wk = wk.with_shape(reduction="none")
            per[key] = measure_config(wk, dev, args.steps, args.warmup, peaks, peak_src,
                                      with_cpu=not args.no_cpu_baseline, **opts)
            print(f"per_config {key}: {per[key]['ms_per_step']} ms/step", file=sys.stderr,
                  flush=True)
        out["per_config"] = per
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
