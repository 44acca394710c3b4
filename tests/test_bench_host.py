"""Host logic of bench.py that needs no GPU: the code-only source hash that keys the recorded
DRAM traffic, and the traffic lookup."""
import bench


def test_code_only_ignores_comments_and_blank_lines():
    a = "int f(int x) // doubles\n{\n    /* the\n       body */\n    return 2 * x;\n}\n"
    b = "int f(int x)\n{\n\n    return 2 * x;   \n}\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_only_sees_code_changes():
    a = "int f(int x) { return 2 * x; } // same comment\n"
    b = "int f(int x) { return 3 * x; } // same comment\n"
    assert bench._code_only(a) != bench._code_only(b)


def test_kernel_source_hash_is_stable_and_short():
    h = bench.kernel_source_hash()
    assert h == bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0


def test_recorded_traffic_is_an_int_or_none():
    for w in ("decode", "prefill", "no-such-workload"):
        v = bench.recorded_traffic(w)
        assert v is None or (isinstance(v, int) and v > 0)
    assert bench.recorded_traffic("no-such-workload") is None
