"""The traffic record is keyed to the scan kernel's device sources by a hash of their code:
comments and whitespace do not count, any change of the code does."""
import bench


def test_comments_and_whitespace_do_not_count():
    a = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    b = "/* the successor */\nint f(int x)\n{\n    return x + 1;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_changes_count():
    a = "int f(int x) { return x + 1; }"
    b = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) != bench._code_only(b)


def test_block_comment_spanning_lines_is_dropped():
    assert bench._code_only("a /* x\n y // z\n */ b") == "a b"
