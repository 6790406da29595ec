"""Host logic of the benchmark (no GPU): the captured DRAM traffic of the fused
kernel is reported only for the kernel code it was measured on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    h = tmp_path / "h.cuh"
    a.write_text("int f(int x) {\n    return x + 1;  // add one\n}\n")
    b.write_text("// header comment\n\nint f(int x) {\n    return x + 1;\n}\n\n")
    c.write_text("int f(int x) {\n    return x + 2;\n}\n")
    h.write_text("#define N 4\n")
    assert bench.code_hash([str(a)]) == bench.code_hash([str(b)])
    assert bench.code_hash([str(a)]) != bench.code_hash([str(c)])
    # an included header and the compiler flags are part of the key
    assert bench.code_hash([str(a), str(h)]) != bench.code_hash([str(a)])
    assert bench.code_hash([str(a)], "-O3") != bench.code_hash([str(a)], "-O2")


def test_fused_traffic_only_for_the_captured_code(monkeypatch):
    per_layer = bench.FUSED_TRAFFIC["bytes_per_layer"]
    if per_layer is not None and bench.fused_code_hash() == bench.FUSED_TRAFFIC["code_sha256"]:
        assert bench.fused_traffic(30) == int(per_layer * 30)
        # traffic at least the algorithmic bytes of a layer's weights (nothing skipped)
        assert per_layer >= bench.BYTES["layer"] / bench.L * 0.99
    monkeypatch.setitem(bench.FUSED_TRAFFIC, "code_sha256", "0" * 64)
    monkeypatch.setitem(bench.FUSED_TRAFFIC, "bytes_per_layer", 1.0)
    assert bench.fused_traffic(30) is None


def test_spread_of_step_times():
    sp = bench.spread([1.0, 2.0, 3.0, 4.0, 100.0])
    assert sp["median_ms"] == 3.0 and sp["n"] == 5
    assert sp["p10_ms"] <= sp["median_ms"] <= sp["p90_ms"]
