"""Host-side logic of bench.py that needs no GPU."""

import bench


def test_source_digest_ignores_comments_and_whitespace_only():
    """A traffic figure stays attached to the kernels' code: editing comments
    or whitespace keeps the digest's input, changing code does not."""
    base = 'int f(int a) {  // add one\n  return a + 1; /* done */\n}\nconst char* s = "x//y";\n'
    comments = '/* header */\nint f(int a) {\n  // add one to a\n      return a + 1;\n}\n\nconst char* s = "x//y";\n'
    code = 'int f(int a) {  // add one\n  return a + 2; /* done */\n}\nconst char* s = "x//y";\n'
    literal = 'int f(int a) {  // add one\n  return a + 1; /* done */\n}\nconst char* s = "x/y";\n'
    assert bench._code_only(base) == bench._code_only(comments)
    assert bench._code_only(base) != bench._code_only(code)
    assert bench._code_only(base) != bench._code_only(literal)
    assert bench._code_only("char c = '\\'';  // quote\nint x;") == "char c = '\\'';\nint x;"

