"""bench.py ties the committed ncu traffic figures to the NS kernel's code: an edit of its
comments keeps them, an edit of its code drops them (the bench line then reports null)."""
import json

import bench


def _tree(tmp_path, body):
    for rel in bench.NS_GEMM_SOURCES:
        path = tmp_path / rel
        path.parent.mkdir(parents=True, exist_ok=True)
        path.write_text(body)


def test_kernel_hash_follows_code_not_comments(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _tree(tmp_path, "int f(int x) {\n  return x + 1;  // one more\n}\n")
    h0 = bench.kernel_hash()
    _tree(tmp_path, "/* a new note */\nint f(int x)   {\n  return x + 1;   // one more, said again\n}\n")
    assert bench.kernel_hash() == h0
    _tree(tmp_path, "int f(int x) {\n  return x + 2;  // one more\n}\n")
    assert bench.kernel_hash() != h0


def test_profiled_traffic_needs_the_same_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _tree(tmp_path, "int f();\n")
    (tmp_path / "profiles").mkdir()
    rec = {"kernel_sha": bench.kernel_hash(), "workloads": {"4": {"bytes_per_launch": 123.0}}}
    (tmp_path / "profiles" / "ns_gemm_traffic.json").write_text(json.dumps(rec))
    assert bench.profiled_traffic(4) == 123.0
    assert bench.profiled_traffic(5) is None
    _tree(tmp_path, "int g();\n")
    assert bench.profiled_traffic(4) is None
