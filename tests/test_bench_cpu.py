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
    a.write_text("int f(int x) {\n    return x + 1;  // add one\n}\n")
    b.write_text("// header comment\n\nint f(int x) {\n    return x + 1;\n}\n\n")
    c.write_text("int f(int x) {\n    return x + 2;\n}\n")
    assert bench.code_hash(str(a)) == bench.code_hash(str(b))
    assert bench.code_hash(str(a)) != bench.code_hash(str(c))


def test_fused_traffic_only_for_the_captured_code(monkeypatch):
    src = os.path.join(ROOT, "bit_expert_streaming_layer_b300", "csrc", "tf_fused.cu")
    per_layer = bench.FUSED_TRAFFIC["bytes_per_layer"]
    if bench.code_hash(src) == bench.FUSED_TRAFFIC["code_sha256"]:
        assert bench.fused_traffic(30) == int(per_layer * 30)
        # traffic at least the algorithmic bytes of a layer's weights (nothing skipped)
        assert per_layer >= bench.BYTES["layer"] / bench.L * 0.99
    monkeypatch.setitem(bench.FUSED_TRAFFIC, "code_sha256", "0" * 64)
    assert bench.fused_traffic(30) is None
