"""Host-side helpers of bench.py that decide whether a committed ncu summary
still describes the kernel: the source hash ignores comments and blank lines
but nothing else."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def test_code_text_drops_comments_and_blank_lines():
    src = 'int a = 1;  // one\n\n/* block\n comment */ int b = 2;\n   \nint c = 3; /* x */\n'
    assert bench.code_text(src) == "int a = 1;\n int b = 2;\nint c = 3;"


def test_code_text_keeps_comment_markers_inside_strings():
    src = 'asm("add.u32 %0, %1; // not a comment");\nint x; // gone\n'
    assert bench.code_text(src) == 'asm("add.u32 %0, %1; // not a comment");\nint x;'
    src2 = 'const char* s = "a\\"/*b*/\\"";\n'
    assert bench.code_text(src2) == 'const char* s = "a\\"/*b*/\\"";'


def test_code_change_changes_hash_but_comment_change_does_not(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = tmp_path / "k.cu"
    f.write_text("int f() { return 1; }  // v1\n")
    h1 = bench.source_hash(["k.cu"])
    f.write_text("// header\nint f() { return 1; }  // v2\n\n")
    assert bench.source_hash(["k.cu"]) == h1
    f.write_text("int f() { return 2; }\n")
    assert bench.source_hash(["k.cu"]) != h1


def test_committed_profiles_name_known_bench_keys():
    pdir = os.path.join(ROOT, "profiles")
    keys = set()
    for name in os.listdir(pdir):
        text = open(os.path.join(pdir, name), encoding="utf-8").read()
        for line in text.splitlines():
            if line.startswith("bench_key:"):
                keys.add(line.split(":", 1)[1].strip())
    assert {"prefill_llama3_t8192_causal", "decode_b64_tk4096"} <= keys
