"""Host-side helpers of bench.py: the source hash that keys stored profiler
counters ignores comments and whitespace but not code, and a stored DRAM
traffic figure is found only under the current hash."""
import bench


def test_code_text_drops_comments_and_whitespace():
    src = "int a; // one\n/* two\n   lines */ int  b;\n\tint c; /* x */"
    assert bench.code_text(src) == "int a; int b; int c;"


def test_code_text_keeps_code_changes():
    assert bench.code_text("x = 1; // n") != bench.code_text("x = 2; // n")


def test_stored_traffic_only_for_the_current_sources():
    # the committed figures were taken on the current kernels' code
    assert bench.stored_traffic("gemm_f16_1024x1024x2048") is not None
    assert bench.stored_traffic("no_such_kernel_key") is None
