"""Host-side helpers of bench.py, without a GPU: the comment stripping behind
the kernel-source hash that ties profiles/dram_traffic.json to the kernels
it was measured on, and the traffic lookup."""
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
