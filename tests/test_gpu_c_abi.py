"""The C ABI from C: tests/c_abi/roundtrip.c is compiled with gcc against
include/flce.h, linked with libflce.so and the CUDA runtime, and run on one
seeded problem (ragged N, V and H tails, 10 % ignored rows, mean reduction,
ignored rows left out). Its outputs are compared with the fp64 oracle under
the bf16 tolerances of tests/_parity.py. No Python or torch code runs in the
C process."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from _parity import (TOL, assert_grad_close, assert_rows_close, assert_scalar_close, ce_row_ops,
                     grad_kappas, row_floor)
from linear_cross_entropy_vocab_gb300 import native_build
from linear_cross_entropy_vocab_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _bf16_bytes(t: torch.Tensor) -> bytes:
    return t.contiguous().view(torch.int16).numpy().tobytes()


def _bf16_from(buf: bytes, shape) -> torch.Tensor:
    a = np.frombuffer(buf, dtype=np.int16).copy()
    return torch.from_numpy(a).view(torch.bfloat16).reshape(shape)


def test_c_program_roundtrip(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib = native_build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = tmp_path / "roundtrip"
    cmd = ["gcc", "-std=c99", "-O1", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(HERE, "c_abi", "roundtrip.c"),
           "-o", str(exe), "-L", os.path.dirname(lib), "-lflce",
           "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{os.path.dirname(lib)}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    w = Workload("c_abi", 300, 136, 1000, "bf16", ignore_frac=0.1)
    x = make_inputs(w)
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([w.n, w.h, w.v, w.ignore_index], dtype=np.int64).tobytes())
        f.write(_bf16_bytes(x["hidden"]))
        f.write(_bf16_bytes(x["weight"]))
        f.write(x["targets"].numpy().astype(np.int64).tobytes())
    r = subprocess.run([str(exe), str(inp), str(out)], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = open(out, "rb").read()
    loss = np.frombuffer(raw[0:4], np.float32)[0]
    n_valid = int(np.frombuffer(raw[4:8], np.int32)[0])
    metrics = np.frombuffer(raw[8:16], np.float32)
    off = 16
    lse = torch.from_numpy(np.frombuffer(raw[off:off + 4 * w.n], np.float32).copy())
    off += 4 * w.n
    gh = _bf16_from(raw[off:off + 2 * w.n * w.h], (w.n, w.h))
    off += 2 * w.n * w.h
    gw = _bf16_from(raw[off:off + 2 * w.v * w.h], (w.v, w.h))

    args = (x["hidden"], x["weight"], x["targets"], None, w.ignore_index, 1.0, None, "mean")
    ref = oracle.forward(*args)
    gref = oracle.backward(*args, 1.0, lse=ref["lse"], magnitudes=True)
    tol = TOL["bf16"]
    nv = ref["n_valid"]
    assert n_valid == nv
    floor = row_floor(w.h, ce_row_ops(ref))
    valid = ref["valid"]
    assert_scalar_close("loss", float(loss), ref["loss_out"], tol["loss_rel"],
                        float(floor[valid].sum()) / nv, float(ref["loss"][valid].sum()) / nv, nv)
    assert abs(float(metrics[1]) - ref["entropy_mean"]) <= tol["ent_rel"] * ref["entropy_mean"]
    assert_rows_close("lse_rows", lse, ref["lse"], tol["loss_rel"], valid, floor)
    kap = grad_kappas(w)
    assert_grad_close("grad_hidden", gh, gref["grad_hidden"], tol, gref["grad_hidden_mag"],
                      kap["grad_hidden"])
    assert_grad_close("grad_weight", gw, gref["grad_weight"], tol, gref["grad_weight_mag"],
                      kap["grad_weight"])
