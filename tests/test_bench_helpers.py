"""Host-side helpers of bench.py: the profile key ignores comments and
whitespace but not code, and the read-probe reference is keyed the same way."""
import bench


def test_code_only_drops_comments_and_whitespace():
    a = "int f(int x) {\n    return x + 1; // one more\n}\n/* block\n comment */\n"
    b = "int f(int x)\n{ return x + 1; }\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_only_keeps_code_changes():
    a = "int f(int x) { return x + 1; }"
    b = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) != bench._code_only(b)


def test_profile_keys_match_the_committed_sources():
    """The committed ncu summaries describe the kernels as they are now (their
    traffic figures are reported only then)."""
    assert bench.profiled_traffic(bench.PROFILE_SUMMARY, "uniform8") is not None
    assert bench.profiled_traffic(bench.W4_PROFILE_SUMMARY, "w4a16", bench.W4_SOURCES) is not None
