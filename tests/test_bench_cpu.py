"""bench.py bookkeeping on CPU: the kernel-code hash that keys the recorded
ncu traffic, and the traffic lookup."""
import bench


def test_code_hash_ignores_comments_and_blank_lines():
    a = "int f(int x) {\n  return x + 1;\n}\n"
    b = "// f: the successor\nint f(int x) {  /* one more */\n\n  return x + 1;  // done\n}\n"
    assert bench.code_hash(a) == bench.code_hash(b)
    assert bench.code_hash(a) != bench.code_hash(a.replace("+ 1", "+ 2"))


def test_traffic_is_read_only_for_the_current_kernel_code(tmp_path, monkeypatch):
    f = tmp_path / "traffic.txt"
    f.write_text(f"# comment: line\nkernel_code_sha256_16: {bench.kernel_hash()}\n"
                 "dram_bytes_per_launch: 123456\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.read_traffic() == 123456.0
    f.write_text("kernel_code_sha256_16: 0000000000000000\ndram_bytes_per_launch: 123456\n")
    assert bench.read_traffic() is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.txt"))
    assert bench.read_traffic() is None
