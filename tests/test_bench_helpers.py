"""Host-side helpers of bench.py: the key that ties a committed ncu summary to
the kernel sources ignores comments and whitespace but not code."""
import bench


def test_code_only_drops_comments_and_whitespace():
    a = "int f(int x) {\n    return x + 1; // one more\n}\n/* block\n comment */\n"
    b = "int f(int x)\n{ return x + 1; }\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_only_keeps_code_changes():
    a = "int f(int x) { return x + 1; }"
    b = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) != bench._code_only(b)


def test_profiled_traffic_scales_a_smaller_case(tmp_path):
    """A profile taken on a smaller case of the workload reports its DRAM
    bytes scaled by the algorithmic bytes of the launch being reported; a
    summary of older sources, or of another workload, reports nothing."""
    import json
    p = tmp_path / "prof.json"
    base = {"workload": "churn", "source_hash": bench.kernel_source_hash(),
            "dram_bytes_per_launch": 1_030_000, "algorithmic_bytes_per_launch": 1_000_000,
            "scaled_from_smaller_case": True}
    p.write_text(json.dumps(base))
    assert bench.profiled_traffic(str(p), "churn", units=4_000_000) == 4_120_000
    assert bench.profiled_traffic(str(p), "uniform8", units=4_000_000) is None
    p.write_text(json.dumps(dict(base, source_hash="0" * 16)))
    assert bench.profiled_traffic(str(p), "churn", units=4_000_000) is None
    p.write_text(json.dumps(dict(base, scaled_from_smaller_case=False)))
    assert bench.profiled_traffic(str(p), "churn", units=4_000_000) == 1_030_000
