"""bench.py reports an ncu traffic figure only while the kernel's code is the code it was taken
on.  The comparison hashes the sources without their comments: these tests check that comments
and blank space drop out, that string literals (where // is not a comment) stay, and that any
change to the code itself changes the hash."""
import importlib.util
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_sources_under_test",
                                                  os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_comments_and_blank_space_drop_out():
    b = _bench()
    src = ('int a = 1;  // the count\n'
           '/* a block\n   comment */ const char* s = "// kept"; char c = \'/\';\n'
           '\n'
           '   x   =  2 ;   \n')
    assert b.code_text(src) == 'int a = 1;\nconst char* s = "// kept"; char c = \'/\';\nx = 2 ;'
    assert b.code_text(src.replace("the count", "how many")) == b.code_text(src)
    assert b.code_text(src.replace("x   =  2", "x = 3")) != b.code_text(src)
    # an escaped quote does not end the literal
    assert b.code_text('s = "a\\" // b"; // c') == 's = "a\\" // b";'


def test_every_kernel_has_a_source_hash():
    b = _bench()
    for kernel in b.KERNEL_SOURCES:
        h = b.sources_sha256(kernel)
        assert len(h) == 64 and int(h, 16) >= 0
