"""Host-side pieces of bench.py on CPU: the kernel-source digest that keys the
stored DRAM counters ignores comments and whitespace but not code."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

SRC = """// header comment
__global__ void k(float* y) {   /* block
   comment */
  y[threadIdx.x] = 1.0f;  // trailing
}
"""


def test_digest_ignores_comments_and_whitespace():
    a = bench.code_digest(SRC)
    b = bench.code_digest(SRC.replace("// header comment", "// another comment")
                          .replace("/* block\n   comment */", "")
                          .replace("  y[", "      y["))
    assert a == b


def test_digest_sees_code_changes():
    a = bench.code_digest(SRC)
    assert bench.code_digest(SRC.replace("1.0f", "2.0f")) != a
    assert bench.code_digest(SRC.replace("threadIdx.x", "threadIdx.y")) != a

