"""Host-side helpers of bench.py: the source hash that keys stored profiler
counters ignores comments and whitespace but not code, and a stored DRAM
traffic figure is found only under a matching kernel key and hash."""
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
