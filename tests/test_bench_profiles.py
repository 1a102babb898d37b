"""The benchmark's link to the committed ncu summaries (CPU only): a summary's DRAM traffic is used
only while the device code it was taken on is unchanged, and comments do not count as code."""
import bench


def test_code_only_drops_comments_and_keeps_literals():
    src = ('int a = 1;  // the count\n'
           '/* a block\n   comment */ const char* s = "// kept"; char q = \'\\\'\';\n'
           '\n'
           'asm("add.f32 %0, %1, %2; // in a string");  /* tail */\n')
    out = bench.code_only(src)
    assert "the count" not in out and "block" not in out and "tail" not in out
    assert '"// kept"' in out and "'\\''" in out and '"add.f32 %0, %1, %2; // in a string"' in out
    assert "\n\n" not in out


def test_traffic_is_reported_only_for_the_code_it_was_taken_on(tmp_path, monkeypatch):
    csrc = tmp_path / "row_wise_online_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    kernel = csrc / "k.cu"
    kernel.write_text("__global__ void k() { int x = 1; }  // v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash(["k.cu"])
    (tmp_path / "profiles" / "k_test__w.md").write_text(
        f"dram_bytes_per_launch: 12345\nsource_files: k.cu\nsource_hash: {h}\n")
    assert bench.profiled_traffic("k_test", "w") == 12345
    kernel.write_text("/* reworded */ __global__ void k() { int x = 1; }  // v2\n")
    assert bench.profiled_traffic("k_test", "w") == 12345  # comments only
    kernel.write_text("__global__ void k() { int x = 2; }\n")
    assert bench.profiled_traffic("k_test", "w") is None  # the code changed
