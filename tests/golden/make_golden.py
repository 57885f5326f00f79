"""Writes tests/golden/tiny_oracle.json: a tiny problem's inputs and the fp64
oracle's outputs for it. Calls only ``oracle/`` (and the seeded input
generator); no value here comes from the CUDA path.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
from linear_cross_entropy_vocab_gb300.workloads import Workload, make_inputs  # noqa: E402

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


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(path, "w") as fh:
        json.dump(build(), fh, indent=1)
    print("wrote", path)
