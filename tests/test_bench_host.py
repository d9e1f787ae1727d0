"""Host-side helpers of bench.py (no GPU): the source fingerprint that keys the recorded
DRAM-traffic capture to the kernel code it was taken on."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    b = _bench()
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {\n  return x + 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("// a comment\nint f(int x) {  // trailing note\n\n  return x + 1;\n}\n\n")
    assert b.code_hash(str(a)) == b.code_hash(str(c))


def test_code_hash_sees_code_changes(tmp_path):
    b = _bench()
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {\n  return x + 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert b.code_hash(str(a)) != b.code_hash(str(c))


def test_traffic_only_for_the_captured_batch():
    b = _bench()
    # the capture holds for the benchmark batch only; any other T reports no traffic
    assert b.traffic_per_launch(4096) is None
    assert b.traffic_per_launch(b.TRAFFIC_CAPTURE["T"]) in (None, b.TRAFFIC_CAPTURE["bytes"])
