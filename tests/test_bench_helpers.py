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
