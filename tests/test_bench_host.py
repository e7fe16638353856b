"""Host logic of bench.py that needs no GPU: the code hash that ties a
committed ncu summary to the kernel source it was taken on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // trailing\n'
           '/* block\n   comment */ const char* s = "x//y/*z*/";\n'
           "char q = '\\''; char r = '/';\n"
           '\n'
           '   \n'
           'a++; /**/ b--;\n')
    out = bench._strip_comments(src)
    assert out == ('int a = 1;\n const char* s = "x//y/*z*/";\n'
                   "char q = '\\''; char r = '/';\n"
                   'a++;  b--;')


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "k.cu").write_text("// header\nint f() { return 1; }  // one\n")
    h0 = bench._source_hash(["k.cu"])
    (tmp_path / "k.cu").write_text("/* a new header */\n\nint f() { return 1; }\n")
    assert bench._source_hash(["k.cu"]) == h0
    (tmp_path / "k.cu").write_text("int f() { return 2; }\n")
    assert bench._source_hash(["k.cu"]) != h0
