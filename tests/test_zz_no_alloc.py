"""vsa_bwd_no_alloc: the backward for callers that cannot allocate device memory (a host framework
that owns all device memory, or a fixed memory budget with no room for a per-call workspace).

It takes no workspace; the library's static scratch array stands in for it.  Called through the
C ABI twice in a row, it must give the same gradients as vsa_bwd with a caller workspace, within
the tolerance the other GPU tests use, and it must refuse shapes whose scratch would not fit.
This file is collected last so that a run stopping at the first failure has already run every
other test; it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

from block_sparse_video_tok_gb300 import workloads as wl
from tests.parity import to_device

pytestmark = pytest.mark.gpu

MAX_BYTES = 32 * 1024 * 1024  # VSA_BWD_NO_ALLOC_MAX_WORKSPACE_BYTES


@pytest.fixture(scope="module")
def vsa():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from block_sparse_video_tok_gb300 import build
    build.build()
    from block_sparse_video_tok_gb300 import vsa as binding
    return binding


def _close(name, got, ref, rel_max=1e-2, mean_rel=1e-3):
    g, r = got.float(), ref.float()
    assert torch.isfinite(g).all(), name
    d = (g - r).abs()
    rm = d.max().item() / max(r.abs().max().item(), 1e-30)
    mr = d.mean().item() / max(r.abs().mean().item(), 1e-30)
    assert rm <= rel_max and mr <= mean_rel, "%s: %.3e %.3e" % (name, rm, mr)


def test_no_alloc_backward_matches_the_workspace_backward(vsa):
    case = wl.make_case(1, 2, 16, 5, vbs="ragged32", seed=31, kv_pool=list(range(14)))
    B, H, S, nb = case["B"], case["H"], case["S"], case["nb"]
    assert vsa.vsa_bwd_workspace_bytes(B, H, S) <= MAX_BYTES
    dev = to_device(case)
    o, lse = vsa.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["q2k_idx"], dev["q2k_num"], dev["vbs"],
                         case["sm_scale"])
    k2q_idx, k2q_num = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], nb)
    args = (dev["do"], dev["q"], dev["k"], dev["v"], o, lse, k2q_idx, k2q_num, dev["vbs"],
            case["sm_scale"])
    ref = vsa.vsa_bwd(*args)
    torch.cuda.synchronize()
    for call in range(2):
        # Outputs start as NaN so that any element the call does not write shows up.
        outs = [torch.full_like(dev["q"], float("nan")) for _ in range(3)]
        got = vsa.vsa_bwd_no_alloc(*args, dq=outs[0], dk=outs[1], dv=outs[2])
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            _close("call %d %s" % (call, name), g, r)
        # dK and dV involve no atomics: identical bits.
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


def test_no_alloc_rejects_shapes_that_do_not_fit(vsa):
    lib = vsa.lib()
    p = ctypes.c_void_p(0x100000)
    too_big = vsa.make_shape(1, 8, 4096)        # needs about 50 MB of scratch
    assert vsa.vsa_bwd_workspace_bytes(1, 8, 4096) > MAX_BYTES
    args = [p] * 8 + [64, p, 0.088, too_big, p, p, p, None]
    assert lib.vsa_bwd_no_alloc(*args) == 3     # VSA_ERR_WORKSPACE, nothing enqueued
    bad_dim = vsa.make_shape(1, 2, 4096, 64)
    args[11] = bad_dim
    assert lib.vsa_bwd_no_alloc(*args) == 2     # VSA_ERR_UNSUPPORTED, as vsa_bwd reports


def test_no_alloc_reports_device_errors(vsa):
    """The error word of a no-allocation call lives in the library's scratch array; the companion
    entry point reads it back.  A k2q id outside [0, nb) is skipped and reported; a clean call
    that follows reports nothing (each call clears the word)."""
    case = wl.make_case(1, 2, 8, 3, vbs="ragged32", seed=32)
    nb = case["nb"]
    dev = to_device(case)
    o, lse = vsa.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["q2k_idx"], dev["q2k_num"], dev["vbs"],
                         case["sm_scale"])
    k2q_idx, k2q_num = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], nb)
    torch.cuda.synchronize()
    args = (dev["do"], dev["q"], dev["k"], dev["v"], o, lse)
    dirty_idx, dirty_num = k2q_idx.clone(), k2q_num.clone()
    j = int(torch.nonzero(k2q_num[0, 0] < nb - 1)[0])
    n = int(k2q_num[0, 0, j])
    dirty_idx[0, 0, j, n] = nb + 3          # one more slot, with an id past the last block
    dirty_num[0, 0, j] = n + 1
    vsa.vsa_bwd_no_alloc(*args, dirty_idx, dirty_num, dev["vbs"], case["sm_scale"])
    bits = vsa.vsa_bwd_no_alloc_device_error()
    assert bits & vsa.DEVERR_K2Q_ID and not bits & vsa.DEVERR_TIMEOUT, hex(bits)
    vsa.vsa_bwd_no_alloc(*args, k2q_idx, k2q_num, dev["vbs"], case["sm_scale"])
    assert vsa.vsa_bwd_no_alloc_device_error() == 0
