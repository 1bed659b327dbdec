"""The committed ncu summaries (profiles/) against what bench.py reads from them.

bench.py reports a kernel's DRAM traffic from profiles/<kind>_<workload>.txt only while the
summary's source_sha256 matches the hash of that kernel's sources; these checks keep the
summaries well formed and the kernel-kind mapping unambiguous. No GPU needed."""
import glob
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUMMARIES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.txt")))


def test_there_are_summaries():
    assert SUMMARIES


def test_kernel_kinds_take_the_longest_prefix():
    assert bench._kernel_kind("decode_i8_llama3_70b_b8_8k") == "decode_i8"
    assert bench._kernel_kind("decode_llama3_70b_b8_8k") == "decode"
    assert bench._kernel_kind("inject_i8_llama3_8b_b32") == "inject_i8"
    assert bench._kernel_kind("inject_llama3_8b_b32") == "inject"
    assert bench._kernel_kind("copy_blocks_mixed_b64_loguniform") == "copy_blocks"
    assert bench._kernel_kind("prefill_llama3_70b_b8_8k") == "prefill"
    assert bench._kernel_kind("combine_llama3_8b_b32") == ""


def test_every_summary_names_its_command_sources_and_traffic():
    for path in SUMMARIES:
        text = open(path).read()
        tag = os.path.basename(path)[:-4]
        kind = bench._kernel_kind(tag)
        assert kind, f"{tag}: no kernel kind"
        lines = dict(ln.split(":", 1) for ln in text.splitlines() if ":" in ln)
        assert "command" in lines and "ncu " in lines["command"], tag
        assert "--clock-control none" in text, tag
        assert float(lines["dram_bytes_per_launch"]) > 0, tag
        assert len(lines["source_sha256"].strip()) == 16, tag
        files = [f.strip() for f in lines["source_files"].split(",")]
        assert files == sorted(set(bench._KERNEL_SOURCES[kind] + bench._COMMON_SOURCES)), tag
        # the summaries are taken on the 2-layer compact copy, one kernel per capture
        assert "--layers 2 --compact-pool" in text, tag


def test_a_stale_summary_reports_no_traffic(tmp_path, monkeypatch):
    src = next(p for p in SUMMARIES if os.path.basename(p).startswith("decode_llama3"))
    text = open(src).read()
    stale = "\n".join("source_sha256: 0000000000000000" if ln.startswith("source_sha256:")
                      else ln for ln in text.splitlines())
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / os.path.basename(src)).write_text(stale)
    (tmp_path / "paged_kv_cache_inject_gb300").mkdir()
    os.symlink(os.path.join(ROOT, "paged_kv_cache_inject_gb300", "csrc"),
               tmp_path / "paged_kv_cache_inject_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic_from_profile(os.path.basename(src)[:-4]) is None


def test_the_hash_follows_code_not_comments():
    code = 'int f(int x) { return x + 1; }\nconst char *s = "a // b";\n'
    commented = ('// a new comment\nint f(int x) {  /* inline */ return x + 1; }\n'
                 'const char *s = "a // b";   // tail\n')
    assert bench._code_only(code) == bench._code_only(commented)
    assert bench._code_only(code) != bench._code_only(code.replace("x + 1", "x + 2"))
    # a comment marker inside a string literal is code
    assert bench._code_only('s = "/* x */";') != bench._code_only('s = "";')
