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


def test_recorded_traffic_matches_the_current_decode_sources():
    rec = bench.recorded_traffic("k_w4a16_gemv", bench.source_digest(bench.DECODE_SOURCES))
    assert rec is not None and rec["dram_bytes_per_step"] > 0
