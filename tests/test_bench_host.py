"""Host-side pieces of bench.py that need no GPU."""

import bench


def test_code_tokens_ignore_comments_and_blank_space_only():
    a = "int f(int x) { // add one\n  return x + 1; /* done */ }\n#define A 1\n"
    b = "/* header */\nint f(int x)   {\n\n return x + 1;  }\n#define A 1 // note\n"
    assert bench.code_tokens(a) == bench.code_tokens(b)
    # a change of code, of a literal, or of where a preprocessor line ends counts
    assert bench.code_tokens(a) != bench.code_tokens(a.replace("x + 1", "x + 2"))
    s = 'const char* p = "// kept /* kept */ \\" kept";'
    assert bench.code_tokens(s) == s
    assert bench.code_tokens("char c = '\"'; int y;") == "char c = '\"'; int y;"
    assert bench.code_tokens("#define A 1\n#define B 2") != \
        bench.code_tokens("#define A 1 #define B 2")


def test_kernel_source_digest_is_a_sha256():
    d = bench.kernel_source_digest()
    assert len(d) == 64 and int(d, 16) >= 0
