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
