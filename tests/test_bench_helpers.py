"""Host-side helpers of bench.py (no GPU): the kernel-source hash that ties
the committed ncu traffic figures to the sources they were taken from."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sources():
    out = {}
    for f in bench.KERNEL_SOURCES:
        with open(os.path.join(ROOT, "tiled_dense_gemm_gb300", "csrc", f), encoding="utf-8") as fh:
            out[f] = fh.read()
    return out


def test_comment_stripping():
    src = "int a; // one\n/* two\n   lines */ int b;\n\n   \nint c;  \n"
    assert bench.code_without_comments(src) == "int a;\n int b;\nint c;"


def test_hash_ignores_comments_only():
    src = _sources()
    base = bench.kernel_source_hash(lambda f: src[f])
    assert base == bench.kernel_source_hash()
    f0 = bench.KERNEL_SOURCES[0]
    commented = dict(src)
    commented[f0] = "// a new comment line\n" + src[f0].replace("\n", "  \n", 3) + "\n/* trailing */\n"
    assert bench.kernel_source_hash(lambda f: commented[f]) == base
    changed = dict(src)
    changed[f0] = src[f0] + "\nstatic int added_for_the_test;\n"
    assert bench.kernel_source_hash(lambda f: changed[f]) != base

