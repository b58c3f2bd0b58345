"""Host logic of bench.py that needs no GPU: the kernel code hash that ties a DRAM capture to the code
it measured."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_strip_comments_keeps_code_and_strings():
    src = ('int a = 1;  // a line comment\n'
           '/* a block\n   comment */ const char *s = "x // y /* z */";\n'
           '\n'
           "char q = '\"'; char r = '\\''; // after quotes\n"
           'asm("mov.u32 %0, 1;" : "=r"(a));   \n')
    got = bench._strip_comments(src)
    assert got.split("\n") == [
        "int a = 1;",
        ' const char *s = "x // y /* z */";',
        "char q = '\"'; char r = '\\'';",
        'asm("mov.u32 %0, 1;" : "=r"(a));',
    ]


def test_kernel_hash_ignores_comments_only():
    path = os.path.join(ROOT, "recoverable_quantized_kv_gb300", "csrc", "decode.cu")
    with open(path, encoding="utf-8") as fh:
        src = fh.read()
    base = bench._strip_comments(src)
    # a comment edit, an added blank line and trailing blanks leave the code unchanged
    edited = "// a new header line\n" + src.replace("\n", "   \n", 3) + "\n\n/* trailing note */\n"
    assert bench._strip_comments(edited) == base
    # a code edit does not
    i = src.index("constexpr int DEC_SLOTS = 36;")
    changed = src[:i] + "constexpr int DEC_SLOTS = 40;" + src[i + len("constexpr int DEC_SLOTS = 36;"):]
    assert bench._strip_comments(changed) != base
    assert len(bench.kernel_sha()) == 16
