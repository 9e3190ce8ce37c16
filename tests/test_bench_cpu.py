"""Host logic of bench.py that needs no GPU."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_kernel_hash_follows_code_not_comments():
    """The kernel hash that ties a committed DRAM-traffic figure to the
    sources it was measured on changes with the code and not with comments,
    blank lines or trailing blanks; comment markers inside string literals
    are code."""
    src = 'int a = 1;  // one\n/* block\n comment */\nconst char* s = "x//y";\n\n'
    assert bench.code_only(src) == 'int a = 1;\nconst char* s = "x//y";'
    base = {f: "int f() { return 1; }\n" for f in bench.KERNEL_SOURCES}

    def reader(files):
        return lambda name: files[name]

    h0 = bench.kernel_hash(reader(base))
    commented = dict(base)
    commented[bench.KERNEL_SOURCES[0]] = "// a comment\nint f() { return 1; }   /* trailing */\n\n"
    assert bench.kernel_hash(reader(commented)) == h0
    changed = dict(base)
    changed[bench.KERNEL_SOURCES[0]] = "int f() { return 2; }\n"
    assert bench.kernel_hash(reader(changed)) != h0
