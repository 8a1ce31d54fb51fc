"""The bench's host-side contract (CPU only): the reference arm's JSON line
carries every key of the bench line format, and the code hash that keys the stored
DRAM-traffic figures ignores comments but not code."""
import io
import json
import os
import sys
import types
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_line_has_the_contract_keys(monkeypatch):
    calls = []

    def fake_baseline(wl, target_s=15.0):
        calls.append(target_s)
        return {"value": 2.0, "unit": "GB/s", "cores": 4, "kind": "oracle", "sample": "stub"}

    monkeypatch.setattr(bench, "cpu_baseline", fake_baseline)
    import oracle
    monkeypatch.setattr(oracle, "build_oracle", lambda: None)
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.reference_main(types.SimpleNamespace(steps=2, warmup=3, gpus=1))
    assert rc == 0 and len(calls) == 5
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] == 2.0 and line["steps"] == 2 and line["warmup"] == 3
    assert line["e2e"] == {"value": 2.0, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 4
    assert "workload" in line["config"]


def test_code_hash_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("/* header */ int f() { return 1; }  // one\n")
    b = tmp_path / "b.cu"
    b.write_text("// another header\nint f()   {\n  return 1;  /* same code */\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("// header\nint f() { return 2; }\n")
    assert bench.code_sha(str(a)) == bench.code_sha(str(b)) != bench.code_sha(str(c))


def test_stored_traffic_matches_the_current_kernel():
    """profiles/traffic.txt holds figures for the kernel code as it is now."""
    sha = bench.code_sha(os.path.join(ROOT, "kv_cache_segment_gb300", "csrc", "attention.cu"))
    lines = [l.split() for l in open(os.path.join(ROOT, "profiles", "traffic.txt")) if l.startswith("traffic ")]
    assert lines and all(l[3] == sha for l in lines), (sha, lines)
