"""Host-side pieces of bench.py: the traffic record of a captured kernel applies only
while that kernel's source file has the same code as at the capture."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_digest_ignores_comments_and_layout_only():
    code = "int f(int a) {\n  return a + 1;  // one more\n}\n"
    assert bench.code_digest(code) == bench.code_digest("/* header */\nint f(int a) {\n\n    return a + 1;\n}\n")
    assert bench.code_digest(code) != bench.code_digest(code.replace("a + 1", "a + 2"))
    assert bench.code_digest(code) != bench.code_digest(code.replace("return a + 1;", "return a + 1;\n  g();"))


def test_traffic_record_applies_only_to_the_captured_code():
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))["gemm_fold_kernel"]
    src = open(os.path.join(ROOT, "fp8_block_scaled_04_gb300", "csrc", rec["source"])).read()
    same = bench.code_digest(src) == rec["code_sha256"]
    assert bench.kernel_traffic("gemm_fold_kernel") == (float(rec["bytes_per_launch"]) if same else None)
    assert bench.kernel_traffic("no_such_kernel") is None
