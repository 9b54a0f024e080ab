"""Host-side helpers of the benchmark: the kernel-source hash that keys committed DRAM
traffic records ignores comments and layout but not code, and a record is used only while
its hash matches the current sources."""

import bench


def test_code_only_ignores_comments_and_whitespace():
    a = "int f(int x) {  // twice\n  return 2 * x; /* doubled */ }\n"
    b = "int f(int x)\n{\n  /* the same,\n     reworded */ return 2*x;\n}\n"
    c = "int f(int x) { return 3 * x; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_kernel_source_hash_is_stable_and_distinct():
    h = bench.kernel_source_hash("tensor_core")
    assert h == bench.kernel_source_hash("tensor_core") and len(h) == 16
    assert h != bench.kernel_source_hash("cuda_core")


def test_recorded_traffic_needs_the_current_hash(tmp_path, monkeypatch):
    cur = bench.kernel_source_hash("tensor_core")
    f = tmp_path / "traffic.txt"
    f.write_text("# comment\n"
                 f"workload=w1 kernel=tensor_core source_hash={cur} dram_bytes=123 summary=x.md\n"
                 "workload=w2 kernel=tensor_core source_hash=0000000000000000 dram_bytes=456 summary=y.md\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("w1", "tensor_core") == 123
    assert bench.recorded_traffic("w2", "tensor_core") is None  # taken on other sources
    assert bench.recorded_traffic("w3", "tensor_core") is None
    assert bench.recorded_traffic("w1", "cuda_core") is None  # another kernel family's record
