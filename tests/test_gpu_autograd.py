"""GPU: the torch.autograd binding (forward -> inversion -> backward through
block_sparse_attention) against the CPU oracle.  O and the gradients of q, k and v must meet the
parity tolerance of tests/parity.py; the gradients are compared with the oracle backward run on
the oracle's own O (rounded to bf16) and lse, so the check also covers the forward's O and lse
feeding the backward.
"""
import numpy as np
import pytest
import torch

from block_sparse_video_tok_gb300 import workloads as wl
from tests.parity import bf16_round, check_close, f64, oracle_backward, oracle_forward, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attention():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from block_sparse_video_tok_gb300 import build
    build.build()
    from block_sparse_video_tok_gb300.autograd import block_sparse_attention
    return block_sparse_attention


CASES = {
    "tiny": lambda: wl.make_config("tiny"),
    "ragged_batch2": lambda: wl.make_case(2, 2, 9, 3, vbs="ragged32", seed=21),
    "4k_25pct": lambda: wl.make_config("4k_25pct"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_autograd_matches_oracle(attention, name):
    case = CASES[name]()
    o64, lse64 = oracle_forward(case)
    dq64, dk64, dv64 = oracle_backward(case, f64(bf16_round(o64)), lse64)
    dev = to_device(case)
    q, k, v = (dev[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    o = attention(q, k, v, dev["q2k_idx"], dev["q2k_num"], dev["vbs"], case["sm_scale"])
    o.backward(dev["do"])
    torch.cuda.synchronize()
    check_close("o", o.detach(), o64)
    check_close("dq", q.grad, dq64)
    check_close("dk", k.grad, dk64)
    check_close("dv", v.grad, dv64)


def test_autograd_default_scale_and_loss(attention):
    """sm_scale defaults to 1/sqrt(128); a scalar loss drives the same gradients as o.backward(dO)."""
    case = wl.make_case(1, 2, 6, 2, seed=22)
    dev = to_device(case)
    q, k, v = (dev[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    o = attention(q, k, v, dev["q2k_idx"], dev["q2k_num"], dev["vbs"])
    (o.float() * dev["do"].float()).sum().backward()
    g1 = [t.grad.clone() for t in (q, k, v)]
    for t in (q, k, v):
        t.grad = None
    o = attention(q, k, v, dev["q2k_idx"], dev["q2k_num"], dev["vbs"], 128 ** -0.5)
    o.backward(dev["do"])
    for a, b in zip(g1, (q.grad, k.grad, v.grad)):
        d = (a.float() - b.float()).abs().max().item()
        assert d <= 5e-3 * b.float().abs().max().item()
