"""Writes tests/golden/tiny_oracle.json and tests/golden/tiny_kl_oracle.json:
tiny problems' inputs and the fp64 oracles' outputs for them (fused linear
cross-entropy; fused linear KL divergence). Calls only ``oracle/`` (and the
seeded input generators); no value here comes from the CUDA path.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
from linear_cross_entropy_vocab_gb300.workloads import (  # noqa: E402
    Workload, make_inputs, make_teacher_probs)
from oracle import kl_oracle  # noqa: E402

CASES = [
    dict(name="softcap_bias_mean", n=6, h=5, v=7, bias_var=0.3, softcap=2.0,
         logit_scale=0.7, ignore_frac=0.34, reduction="mean"),
    dict(name="plain_sum", n=5, h=4, v=9, bias_var=None, softcap=None,
         logit_scale=1.0, ignore_frac=0.2, reduction="sum"),
]


def build():
    out = {"note": "inputs drawn by the seeded generator (seed 0) at fp32; "
                   "expected values from oracle.forward / oracle.backward in fp64",
           "cases": []}
    for c in CASES:
        w = Workload(c["name"], c["n"], c["h"], c["v"], "f32", bias_var=c["bias_var"],
                     ignore_frac=c["ignore_frac"], logit_scale=c["logit_scale"],
                     softcap=c["softcap"], reduction=c["reduction"])
        x = make_inputs(w)
        args = (x["hidden"], x["weight"], x["targets"], x["bias"], -100,
                c["logit_scale"], c["softcap"], c["reduction"])
        f = oracle.forward(*args)
        g = oracle.backward(*args, 1.0)
        out["cases"].append({
            **c,
            "hidden": x["hidden"].tolist(), "weight": x["weight"].tolist(),
            "bias": None if x["bias"] is None else x["bias"].tolist(),
            "targets": x["targets"].tolist(),
            "loss_rows": f["loss"].tolist(), "lse": f["lse"].tolist(),
            "entropy": f["entropy"].tolist(), "argmax": f["argmax"].tolist(),
            "loss_out": f["loss_out"], "mean_token_accuracy": f["mean_token_accuracy"],
            "entropy_mean": f["entropy_mean"],
            "grad_hidden": g["grad_hidden"].tolist(), "grad_weight": g["grad_weight"].tolist(),
            "grad_bias": None if g["grad_bias"] is None else g["grad_bias"].tolist(),
        })
    return out


KL_CASES = [
    dict(name="kl_bias_labels_batchmean", n=6, h=5, v=7, bias_var=0.3, ignore_frac=0.34,
         temperature=1.5, reduction="batchmean", keep_top=None),
    dict(name="kl_topk_sum", n=5, h=4, v=9, bias_var=None, ignore_frac=0.0,
         temperature=0.7, reduction="sum", keep_top=3),
]


def build_kl():
    out = {"note": "inputs drawn by the seeded generators (seed 0) at fp32; teacher "
                   "probabilities from make_teacher_probs; expected values from "
                   "kl_oracle.forward / kl_oracle.backward in fp64 (eps 1e-10)",
           "cases": []}
    for c in KL_CASES:
        w = Workload(c["name"], c["n"], c["h"], c["v"], "f32", bias_var=c["bias_var"],
                     ignore_frac=c["ignore_frac"])
        x = make_inputs(w)
        q = make_teacher_probs(w, keep_top=c["keep_top"])
        labels = x["targets"] if c["ignore_frac"] > 0 else None
        args = (x["hidden"], x["weight"], q, x["bias"], labels, -100, c["temperature"], 1e-10,
                c["reduction"])
        f = kl_oracle.forward(*args)
        g = kl_oracle.backward(*args, 1.0)
        out["cases"].append({
            **c,
            "hidden": x["hidden"].tolist(), "weight": x["weight"].tolist(),
            "bias": None if x["bias"] is None else x["bias"].tolist(),
            "target_probs": q.tolist(), "labels": None if labels is None else labels.tolist(),
            "loss_rows": f["loss"].tolist(), "lse": f["lse"].tolist(), "qsum": f["qsum"].tolist(),
            "loss_out": f["loss_out"], "n_counted": f["n_counted"],
            "grad_hidden": g["grad_hidden"].tolist(), "grad_weight": g["grad_weight"].tolist(),
            "grad_bias": None if g["grad_bias"] is None else g["grad_bias"].tolist(),
        })
    return out


if __name__ == "__main__":
    here = os.path.dirname(os.path.abspath(__file__))
    for name, data in (("tiny_oracle.json", build()), ("tiny_kl_oracle.json", build_kl())):
        path = os.path.join(here, name)
        with open(path, "w") as fh:
            json.dump(data, fh, indent=1)
        print("wrote", path)
