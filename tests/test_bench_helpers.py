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


def test_main_kernel_profile_follows_the_committed_capture(bench):
    """The roofline's traffic and tensor-pipe figures come from profiles/bwd_main_32k.md only while
    the kernel's code still has the hash recorded there; otherwise both are None."""
    import re
    text = open(os.path.join(ROOT, "profiles", "bwd_main_32k.md")).read()
    recorded = re.search(r"code sha256 at capture: `([0-9a-f]{64})`", text).group(1)
    src = open(os.path.join(ROOT, "block_sparse_video_tok_gb300", "csrc", "bwd_main.cu")).read()
    traffic, tensor = bench.main_kernel_profile("32k_25pct")
    if bench.kernel_code_hash(src) == recorded:
        assert isinstance(traffic, int) and traffic > 0
        assert 0.0 < tensor < 1.0
    else:
        assert traffic is None and tensor is None
