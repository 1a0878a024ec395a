"""Host logic of bench.py that needs no GPU: the kernel source hash behind the
DRAM-traffic record changes with the code and not with comments or layout."""
import importlib.util
import os

from conftest import ROOT


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_strip_comments_keeps_code_and_literals():
    b = _bench()
    src = 'int a; // one\n/* two\n three */ const char* s = "x // y /* z */"; char c = \'"\';\n  float f;'
    assert b.strip_comments(src) == 'int a; const char* s = "x // y /* z */"; char c = \'"\'; float f;'


def test_comment_and_layout_edits_do_not_change_the_stripped_source():
    b = _bench()
    code = "__global__ void k(int* p) {\n  p[0] = 1;  // set\n}\n"
    edited = "/* a new header comment */\n__global__ void k(int* p) {\n\n    p[0] = 1;\n}\n"
    changed = "__global__ void k(int* p) {\n  p[0] = 2;\n}\n"
    assert b.strip_comments(code) == b.strip_comments(edited)
    assert b.strip_comments(code) != b.strip_comments(changed)


def test_every_kernel_file_hashes():
    b = _bench()
    for op, src in b.KERNEL_FILE.items():
        h = b.kernel_source_hash(src)
        assert h is not None and len(h) == 16 and int(h, 16) >= 0, op
