"""Host-side pieces of bench.py that need no GPU."""

import re

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


def _profile_commands():
    """Every `python bench.py ...` command quoted in profiles/ (line
    continuations joined), with its argument list."""
    import glob
    import os
    import re
    import shlex
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for path in sorted(glob.glob(os.path.join(root, "profiles", "*.md"))):
        text = re.sub(r"\\\s*\n\s*", " ", open(path).read())
        for m in re.finditer(r"python bench\.py([^`\n]*)", text):
            tail = re.split(r"\s(?:>|&&|\|)", m.group(1))[0]
            yield os.path.basename(path), shlex.split(tail)


def test_profile_commands_parse_with_the_current_flags():
    seen = 0
    for name, argv in _profile_commands():
        # placeholders such as M,N,K or {cuda,tensor} stand for a sweep
        if any(re.search(r"[A-Z],|\{", a) for a in argv):
            continue
        try:
            bench.build_parser().parse_args(argv)
        except SystemExit:
            raise AssertionError(f"{name}: bench.py {' '.join(argv)} no longer parses")
        seen += 1
    assert seen >= 8
