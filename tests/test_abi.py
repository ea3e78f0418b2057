"""The C ABI without a GPU: libvsa.so builds, loads, exports every function include/vsa.h
declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import math
import os
import re
import shutil

import pytest

from block_sparse_video_tok_gb300 import build as vsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vsa.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="nvcc is needed to build libvsa.so")


@pytest.fixture(scope="module")
def vsa():
    vsa_build.build()
    from block_sparse_video_tok_gb300 import vsa as binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vsa_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(vsa):
    names = declared_functions()
    assert len(names) == 13, names
    lib = vsa.lib()
    for name in names:
        assert hasattr(lib, name), name
        assert name in vsa.SIGNATURES, name


def test_status_strings(vsa):
    assert vsa.status_string(0) == "VSA_OK"
    assert vsa.status_string(3) == "VSA_ERR_WORKSPACE"
    assert vsa.status_string(99) == "VSA_ERR_UNKNOWN"


def test_workspace_sizes(vsa):
    B, H, S = 2, 3, 640
    rows = B * H * S
    bwd = vsa.vsa_bwd_workspace_bytes(B, H, S)
    fwd = vsa.vsa_fwd_workspace_bytes(B, H, S)
    # dQ accumulator (fp32) + four fp16 operand copies dominate the backward workspace.
    assert bwd >= rows * 128 * 4 + 4 * rows * 128 * 2 + rows * 4
    # The forward copies only V to fp16 (S = Q K^T takes the bf16 Q and K as given).
    assert rows * 128 * 2 <= fwd < 2 * rows * 128 * 2
    assert vsa.vsa_bwd_workspace_bytes(B, H, 100) == 0      # S not a multiple of 64
    assert vsa.vsa_bwd_workspace_bytes(B, H, S, 64) == 0    # head_dim 64
    assert vsa.vsa_fwd_workspace_bytes(0, H, S) == 0


def _bwd_args(vsa, shape, ptr=0x100000, ws_bytes=1 << 40, scale=0.088):
    p = ctypes.c_void_p(ptr)
    return [p, p, p, p, p, p, p, p, 8, p, scale, shape, p, p, p, p, ws_bytes, None]


def test_host_side_rejections(vsa):
    lib = vsa.lib()
    good = vsa.make_shape(1, 2, 512)
    # Null pointers.
    null = [None] * 8 + [8, None, 0.1, good] + [None] * 4 + [1 << 40, None]
    assert lib.vsa_bwd(*null) == 1
    # Unsupported head_dim / sequence length.
    assert lib.vsa_bwd(*_bwd_args(vsa, vsa.make_shape(1, 2, 512, 64))) == 2
    assert lib.vsa_bwd(*_bwd_args(vsa, vsa.make_shape(1, 2, 500))) == 2
    # Block size: 64 or 128 (0 read as 64), and S a multiple of it.
    assert lib.vsa_bwd(*_bwd_args(vsa, vsa.make_shape(1, 2, 512, 128, 96))) == 2
    assert lib.vsa_bwd(*_bwd_args(vsa, vsa.make_shape(1, 2, 576, 128, 128))) == 2
    assert lib.vsa_bwd(*_bwd_args(vsa, vsa.make_shape(1, 2, 512, 128, 128), ws_bytes=1024)) == 3
    assert lib.vsa_bwd(*_bwd_args(vsa, vsa.make_shape(1, 2, 512, 128, 0), ws_bytes=1024)) == 3
    # Non-finite softmax scale, bad row stride, misaligned pointer.
    assert lib.vsa_bwd(*_bwd_args(vsa, good, scale=math.inf)) == 1
    bad = _bwd_args(vsa, good)
    bad[8] = 0
    assert lib.vsa_bwd(*bad) == 1
    assert lib.vsa_bwd(*_bwd_args(vsa, good, ptr=0x100008)) == 1
    # Workspace too small.
    assert lib.vsa_bwd(*_bwd_args(vsa, good, ws_bytes=1024)) == 3
    p = ctypes.c_void_p(0x100000)
    assert lib.vsa_invert_indices(p, p, 0, good, p, p, None, None) == 1
    assert lib.vsa_fwd(p, p, p, p, p, 4, p, 0.1, good, p, p, p, 16, None) == 3


def test_host_side_rejections_of_the_helpers(vsa):
    lib = vsa.lib()
    p = ctypes.c_void_p(0x100000)
    good = vsa.make_shape(1, 2, 512)
    assert lib.vsa_work_order(None, 8, good, p, None) == 1        # null counts
    assert lib.vsa_work_order(p, 0, good, p, None) == 1           # max_q_blocks < 1
    assert lib.vsa_work_order(p, 8, vsa.make_shape(1, 2, 500), p, None) == 2
    assert lib.vsa_bwd_no_alloc_device_error(None, None) == 1     # no place for the bits


def test_wait_limit_setting_round_trips(vsa):
    lib = vsa.lib()
    default = 4_000_000_000
    prev = lib.vsa_set_wait_limit_ns(1000)
    assert prev == default
    assert lib.vsa_set_wait_limit_ns(0) == 1000                   # 0 restores the default
    assert lib.vsa_set_wait_limit_ns(0) == default
