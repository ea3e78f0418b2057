"""Host-side helpers of bench.py (no GPU): the kernel-code hash that decides whether the committed
ncu traffic figure still belongs to the main kernel."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


SRC = """// kernel comment
__global__ void k(int* x) {  /* block
  comment */
  x[0] = 1;   // trailing
}
"""


def test_code_hash_ignores_comments_and_spacing(bench):
    h = bench.kernel_code_hash(SRC)
    edited = SRC.replace("// kernel comment", "// another comment\n// over two lines")
    edited = edited.replace("/* block\n  comment */", "/* other */").replace("x[0] = 1;",
                                                                              "x[0]  =  1;")
    assert bench.kernel_code_hash(edited) == h


def test_code_hash_follows_code_changes(bench):
    h = bench.kernel_code_hash(SRC)
    assert bench.kernel_code_hash(SRC.replace("x[0] = 1;", "x[0] = 2;")) != h
    assert bench.kernel_code_hash(SRC.replace("int* x", "int* y")) != h
