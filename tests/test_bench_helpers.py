"""Host-side helpers of bench.py (no GPU): the source digest that keys the
recorded DRAM traffic follows the code, not its comments."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_ignores_comments_not_code():
    a = 'int x = 1;  // one\n/* a block\n   comment */\n\nconst char* s = "a//b /* c */";\n'
    b = 'int x = 1;\nconst char* s = "a//b /* c */";\n'
    c = 'int x = 2;\nconst char* s = "a//b /* c */";\n'
    d = "char q = '\"'; // quote\nint y;\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only(d) == "char q = '\"';\nint y;"


def test_traffic_record_shape():
    """One DRAM figure per decode launch of a step, summing to the step's;
    bench.py reports it only while the digest matches the sources."""
    import json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["k_w4a16_gemv"]
    assert len(rec["source_digest"]) == 16
    assert len(rec["dram_bytes_per_launch"]) == 4
    assert sum(rec["dram_bytes_per_launch"]) == rec["dram_bytes_per_step"]
    assert bench.recorded_traffic("k_w4a16_gemv", "0" * 16) is None


def test_reference_arm_line():
    """`bench.py --impl reference` (the oracle on the host cores; no GPU)
    prints one JSON line in the bench contract, its cpu_baseline and e2e
    describing the same run."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]
