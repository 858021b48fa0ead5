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


def test_reference_arm_reports_what_it_timed(monkeypatch, capsys):
    """The reference arm's line: K x ms_per_step is its timed wall time, and the value is the
    bank-steps those K steps processed (K times the fraction) over that time."""
    import time
    clock = iter([10.0, 10.0 + 0.25 * 3]).__next__     # 3 timed steps of 0.25 s
    monkeypatch.setattr(bench, "oracle_matrix_step", lambda wl, st: None)
    monkeypatch.setattr(bench, "one_matrix_states", lambda wl, seed: [None] * len(wl.banks))
    monkeypatch.setattr(time, "perf_counter", clock)
    args = type("A", (), dict(workload=4, steps=3, warmup=1, gpus=1))()
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["ms_per_step"] * line["steps"] == 750.0
    assert abs(line["value"] - 3 * bench.REF_FRACTION[4] / 0.75) < 1e-12
    assert line["cpu_baseline"]["value"] == line["value"] == line["e2e"]["value"]


def test_reference_windows_cover_each_bank_in_turn():
    """Steps 0 .. 1/f - 1 of the moving window touch every slot of a bank exactly once."""
    for batch, f in ((40, 1 / 8), (24, 1 / 8), (10, 1 / 8), (1, 1 / 8), (96, 1 / 48), (48, 1 / 48)):
        seen = [s for k in range(round(1 / f)) for s in bench.ref_window(batch, f, k)]
        assert sorted(seen) == list(range(batch)), (batch, f)
