"""Host-side pieces of bench.py that need no GPU: the key that ties the recorded DRAM traffic of the
histogram kernel to its code."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_key_ignores_comments_but_not_code():
    src = "int a = 1;  // one\n/* a\n   block */\n\nint b = a + 2;\n"
    same = "// header\nint a = 1;\n\n\nint b = a + 2;  /* trailing */\n"
    other = "int a = 1;\nint b = a + 3;\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)

