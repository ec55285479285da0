"""Host logic of bench.py that needs no GPU: the key that ties the committed ncu traffic
figure to the GEMM kernel's code."""

import bench


def test_strip_comments_keeps_code_only():
    src = "int a = 1; // one\n/* two\n lines */ int   b =\n\t2;  // tail\n"
    assert bench.strip_comments(src) == "int a = 1; int b = 2;"


def test_comment_and_layout_edits_keep_the_key_code_edits_change_it():
    base = "__global__ void k(int *p) {\n  p[0] = 1;  // store\n}\n"
    recommented = "// the kernel\n__global__ void k(int *p) {\n  /* one store */ p[0] = 1;\n}\n"
    changed = "__global__ void k(int *p) {\n  p[0] = 2;\n}\n"
    assert bench.strip_comments(base) == bench.strip_comments(recommented)
    assert bench.strip_comments(base) != bench.strip_comments(changed)

