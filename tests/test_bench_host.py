"""Host helpers of bench.py that need no GPU: the kernel-source hash that
keys the recorded DRAM traffic (profiles/traffic.json) to the sources it was
captured on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_layout():
    src = 'int a = 1;  // trailing note\n/* block\n comment */ int  b = 2;\n'
    assert bench._code_only(src) == "int a = 1; int b = 2;"


def test_code_only_keeps_string_literals():
    src = 'asm("add.rn.f32 %0, %1; // not a comment");  // a comment\nconst char* s = "a \\" /* b";\n'
    assert bench._code_only(src) == 'asm("add.rn.f32 %0, %1; // not a comment"); const char* s = "a \\" /* b";'


def test_code_changes_change_the_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "turboquant_kv_cache_tq_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("int f() { return 1; }  // one\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (csrc / "k.cu").write_text("// a new comment\nint f() {\n  return 1;\n}\n")
    assert bench.kernel_source_hash() == h0
    (csrc / "k.cu").write_text("int f() { return 2; }\n")
    assert bench.kernel_source_hash() != h0
