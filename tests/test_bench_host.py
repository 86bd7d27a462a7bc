"""Host logic of bench.py that needs no GPU: the kernel-code hash that keys a
stored ncu traffic figure ignores comments and whitespace but not code (a
code change makes the benchmark report traffic as null until re-captured)."""
import bench


def test_code_only_drops_comments_and_whitespace_but_keeps_literals():
    src = 'int a = 1; // note\n/* block\n comment */ const char* s = "x // y /* z */";\n'
    assert bench.code_only(src) == 'inta=1;constchar*s="x // y /* z */";'
    assert bench.code_only("char q = '\"'; int b;") == "charq='\"';intb;"


def test_code_hash_sees_code_changes_only():
    a = "int f(int x) {\n    return x + 1;  // one\n}\n"
    b = "int f(int x) {  /* edited comment */\n  return x + 1;\n}\n"
    c = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)

