"""The watchdog of the kernels' pipeline waits, made to fire without planting any defect.

Every wait inside the forward and backward kernels has a time limit (vsa_set_wait_limit_ns).  With
the limit set far below the time a normal wait takes (here 200 ns, against microseconds for a
tile copy), the waits run out: the kernel must report VSA_DEVERR_TIMEOUT in its error word, let
its copies in flight land, free its tensor memory and return, leaving the device usable.  The
same calls with the default limit then give results that pass parity against the oracle.
"""
import numpy as np
import pytest
import torch

from block_sparse_video_tok_gb300 import workloads as wl
from tests.parity import bf16_round, check_close, f64, oracle_backward, oracle_forward, to_device

pytestmark = pytest.mark.gpu

SHORT_NS = 200


@pytest.fixture(scope="module")
def vsa():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from block_sparse_video_tok_gb300 import build
    build.build()
    from block_sparse_video_tok_gb300 import vsa as binding
    return binding


def test_short_wait_limit_reports_timeout_then_recovers(vsa):
    case = wl.make_case(1, 4, 64, 16, vbs="ragged32", seed=61)
    B, H, S, nb = case["B"], case["H"], case["S"], case["nb"]
    dev = to_device(case)
    o64, lse64 = oracle_forward(case)
    o_b = bf16_round(o64)
    lse32 = lse64.astype(np.float32)
    dq64, dk64, dv64 = oracle_backward(case, f64(o_b), lse32.astype(np.float64))
    k2q_idx, k2q_num = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], nb)
    fws = torch.empty(vsa.vsa_fwd_workspace_bytes(B, H, S), dtype=torch.uint8, device="cuda")
    bws = torch.empty(vsa.vsa_bwd_workspace_bytes(B, H, S), dtype=torch.uint8, device="cuda")
    bwd_args = (dev["do"], dev["q"], dev["k"], dev["v"], o_b.cuda(),
                torch.from_numpy(lse32).cuda(), k2q_idx, k2q_num, dev["vbs"], case["sm_scale"])
    torch.cuda.synchronize()
    prev = vsa.vsa_set_wait_limit_ns(SHORT_NS)
    try:
        vsa.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["q2k_idx"], dev["q2k_num"], dev["vbs"],
                    case["sm_scale"], workspace=fws)
        fwd_bits = vsa.vsa_read_device_error(fws)
        vsa.vsa_bwd(*bwd_args, workspace=bws)
        bwd_bits = vsa.vsa_read_device_error(bws)
    finally:
        vsa.vsa_set_wait_limit_ns(prev)
    assert fwd_bits & vsa.DEVERR_TIMEOUT, hex(fwd_bits)
    assert bwd_bits & vsa.DEVERR_TIMEOUT, hex(bwd_bits)
    # The context is intact: the same calls with the normal limit are correct.
    o, lse = vsa.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["q2k_idx"], dev["q2k_num"], dev["vbs"],
                         case["sm_scale"], workspace=fws)
    assert vsa.vsa_read_device_error(fws) == 0
    check_close("o", o, o64)
    outs = [torch.full_like(dev["q"], float("nan")) for _ in range(3)]
    dq, dk, dv = vsa.vsa_bwd(*bwd_args, dq=outs[0], dk=outs[1], dv=outs[2], workspace=bws)
    assert vsa.vsa_read_device_error(bws) == 0
    check_close("dq", dq, dq64)
    check_close("dk", dk, dk64)
    check_close("dv", dv, dv64)
