"""bench.py reports ncu-measured DRAM traffic only for the kernel sources it was
measured on: the committed summary records a digest of those sources."""
import bench


def test_traffic_is_reported_only_for_matching_sources(tmp_path, monkeypatch):
    summary = tmp_path / "summary.txt"
    summary.write_text(f"# header\nkernel_sources_sha256: {bench.kernel_sources_digest()}\n"
                       "dram_bytes_per_launch: 12345\n- kernel_sources_sha256 is explained here\n")
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(summary))
    assert bench.profiled_traffic() == 12345
    summary.write_text("kernel_sources_sha256: 00\ndram_bytes_per_launch: 12345\n")
    assert bench.profiled_traffic() is None
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(tmp_path / "missing.txt"))
    assert bench.profiled_traffic() is None


def test_digest_sees_code_not_comments():
    a = "int f(int x) {  // doubles\n  return 2 * x; /* no overflow here */\n}\n"
    b = "/* header */\nint f(int x) {\n\n  return 2 * x;\n}\n"
    c = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(c)
    s = 'asm("mov.u32 %0, 1; // kept");\n'
    assert bench.strip_comments(s) == s.strip()
