"""Host-side helpers of bench.py: the source hash that keys stored profiler
counters ignores comments and whitespace but not code, and a stored DRAM
traffic figure is found only under a matching kernel key and hash, and the
--timeline summary of kernel stamps."""
import numpy as np

import bench


def test_code_text_drops_comments_and_whitespace():
    src = "int a; // one\n/* two\n   lines */ int  b;\n\tint c; /* x */"
    assert bench.code_text(src) == "int a; int b; int c;"


def test_code_text_keeps_code_changes():
    assert bench.code_text("x = 1; // n") != bench.code_text("x = 2; // n")


def test_stored_traffic_needs_a_matching_key():
    assert bench.stored_traffic("no_such_kernel_key") is None
    v = bench.stored_traffic("gemm_f16_1024x1024x2048")     # None once the kernels' code changes
    assert v is None or v > 0


def test_timeline_rows_relative_to_first_entry():
    """Slots nobody wrote are left out; times are from the earliest entry
    stamp, over the CTAs that wrote the slot; rows of CTAs that did not run
    (entry stamp 0) are ignored."""
    t = np.zeros((4, 64), dtype=np.int64)
    t[0, 0], t[1, 0], t[2, 0] = 1_000_000, 1_002_000, 1_001_000
    t[0, 5], t[1, 5] = 1_010_000, 1_014_000
    t[2, 63] = 1_003_500
    t[3, 5] = 9_999_999_999                  # CTA without an entry stamp
    rows = bench.timeline_rows(t)
    assert [r[0] for r in rows] == [0, 5, 63]
    assert rows[0] == (0, 0.0, 1.0, 2.0)
    assert rows[1] == (5, 10.0, 12.0, 14.0)
    assert rows[2] == (63, 3.5, 3.5, 3.5)
    assert bench.timeline_rows(np.zeros((2, 64), dtype=np.int64)) == []
