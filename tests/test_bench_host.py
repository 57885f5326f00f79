"""Host-side helpers of bench.py, without a GPU: the comment stripping behind
the kernel-source hash that ties profiles/dram_traffic.json to the kernels
it was measured on, the traffic lookup, and the roofline entry of the
dominant kernel (its achieved flops and the peak it is set against)."""
import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_strip_c_comments_keeps_code_and_literals():
    b = _bench()
    src = 'int a = 1; // note\n/* block\n comment */ const char* s = "// kept";\nchar c = \'/\';'
    assert b.strip_c_comments(src) == 'int a = 1; const char* s = "// kept"; char c = \'/\';'
    # a comment edit does not change the stripped text; a code edit does
    assert b.strip_c_comments("x = 1; // a") == b.strip_c_comments("x = 1;   // b c")
    assert b.strip_c_comments("x = 1;") != b.strip_c_comments("x = 2;")
    assert b.strip_c_comments('asm("mov.u32 %0, 1;" : "=r"(r)); /* x */') == \
        'asm("mov.u32 %0, 1;" : "=r"(r));'


def test_traffic_lookup_follows_the_hash(tmp_path, monkeypatch):
    b = _bench()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (tmp_path / "include").mkdir()
    (tmp_path / "include" / "flce.h").write_text("int f(void);\n")
    csrc = tmp_path / "linear_cross_entropy_vocab_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("__global__ void k() {}  // v1\n")
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    rec = {"csrc_sha256": b.kernel_sources_sha256(),
           "workloads": {"w": {"bytes_per_launch": {"fwd_stats": 123}}}}
    (prof / "dram_traffic.json").write_text(json.dumps(rec))
    assert b.measured_traffic("fwd_stats", "w") == 123
    (csrc / "k.cu").write_text("__global__ void k() {}  // v2, comment only\n")
    assert b.measured_traffic("fwd_stats", "w") == 123
    (csrc / "k.cu").write_text("__global__ void k() { return; }\n")
    assert b.measured_traffic("fwd_stats", "w") is None
    assert b.measured_traffic("fwd_stats", "other") is None


PEAKS = {"bf16_tflops": 1856.7, "bf16_tflops_sustained": 1661.6, "sm_max_mhz": 2070.0}


def test_roofline_tensor_peak_follows_the_timed_region():
    """A GEMM role is set against the sustained bf16 peak when the timed region
    lasts a second or more, else against the burst peak; achieved is the
    launch's 2 n h v flops (split over its launches per step) over its average
    duration."""
    b = _bench()
    n, h, v, steps = 8028, 4096, 128256, 60
    # 4 dlogits launches per step, 1.267 ms each
    long = b.roofline_entry("bwd_dlogits", 4 * steps, 4 * steps * 1.267, steps, n, h, v,
                            1200.0, PEAKS, "measured", 152)
    per_launch = 2.0 * n * h * v / 4
    assert long["flops_per_launch"] == per_launch
    assert abs(long["achieved"] - per_launch / 1.267e-3 / 1e12) < 0.1
    assert long["bound"] == "tensor" and long["peak"] == 1661.6
    assert "sustained" in long["peak_kind"]
    assert abs(long["frac"] - long["achieved"] / 1661.6) < 1e-3
    short = b.roofline_entry("bwd_dlogits", 4 * steps, 4 * steps * 1.267, steps, n, h, v,
                             999.0, PEAKS, "measured", 152)
    assert short["peak"] == 1856.7 and "burst" in short["peak_kind"]
    assert short["achieved"] == long["achieved"]


def test_roofline_fused_gradient_role_counts_both_contractions():
    """bwd_grads runs grad_hidden and grad_weight of a chunk in one launch:
    4 n h v flops per step, split over its launches."""
    b = _bench()
    n, h, v, steps = 8028, 4096, 128256, 10
    r = b.roofline_entry("bwd_grads", 5 * steps, 5 * steps * 2.0, steps, n, h, v, 500.0,
                         PEAKS, "measured", 152)
    assert r["flops_per_launch"] == 4.0 * n * h * v / 5
    assert abs(r["achieved"] - 4.0 * n * h * v / 5 / 2.0e-3 / 1e12) < 0.1


def test_roofline_split_roles_use_a_sixth_of_the_bf16_peak():
    """fp32 operands split into three bf16 parts take six bf16 products per
    fp32 product: the split roles count the algorithmic fp32 flops against the
    bf16 peak / 6."""
    b = _bench()
    n, h, v, steps = 8192, 4096, 128256, 3
    r = b.roofline_entry("bwd_grads_split", 18 * steps, 18 * steps * 3.66, steps, n, h, v,
                         380.0, PEAKS, "measured", 152)
    assert r["bound"] == "tensor"
    assert r["peak"] == round(1856.7 / 6, 1)
    assert "/ 6" in r["peak_kind"]
    assert r["flops_per_launch"] == 4.0 * n * h * v / 18
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3


def test_roofline_fp32_roles_use_the_fma_peak():
    """The fp32 (FFMA) roles are ALU-bound: the peak is SMs x 128 lanes x 2 flops
    x the maximum SM clock, whatever the length of the timed region."""
    b = _bench()
    r = b.roofline_entry("bwd_grad_hidden_f32", 3, 3 * 10.8, 3, 4096, 2048, 32000, 120.0,
                         PEAKS, "measured", 152)
    assert r["bound"] == "alu"
    assert r["peak"] == round(152 * 128 * 2 * 2070e6 / 1e12, 1) == 80.5
    assert abs(r["achieved"] - 2.0 * 4096 * 2048 * 32000 / 10.8e-3 / 1e12) < 0.1
    r2 = b.roofline_entry("bwd_grad_hidden_f32", 3, 3 * 10.8, 3, 4096, 2048, 32000, 5000.0,
                          PEAKS, "measured", 152)
    assert r2["peak"] == r["peak"]


def test_roofline_non_gemm_role_has_no_flops():
    b = _bench()
    r = b.roofline_entry("merge_rows", 60, 1.2, 60, 8192, 4096, 128256, 1200.0, PEAKS,
                         "measured", 152)
    assert r["flops_per_launch"] == 0.0 and r["achieved"] == 0.0
