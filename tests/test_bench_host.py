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


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on the host cores and prints
    one JSON line with the arm's keys (the decode mode keeps the sample small)."""
    import json
    import subprocess
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--mode", "decode", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["steps"] == 1 and d["warmup"] >= 3 and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["higher_is_better"] is True and d["config"]["workload"]
