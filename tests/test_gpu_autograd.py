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
    "blk128_ragged": lambda: wl.make_case(1, 2, 6, 2, vbs="ragged65", seed=23, blk=128),
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


def test_saved_k2q_and_caller_k2q_agree(attention):
    """The forward inverts the selection once and saves it; a caller may pass that inversion in
    instead (layers that share one selection).  Both give the same gradients: dK and dV bit for
    bit (no atomics), dQ within 5e-3 of max|dQ| (fp32 partial sums in a varying order)."""
    from block_sparse_video_tok_gb300 import vsa
    case = wl.make_case(1, 3, 24, 6, vbs="ragged32", seed=24)
    dev = to_device(case)
    k2q = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], case["nb"])
    grads = []
    for given in (None, k2q):
        q, k, v = (dev[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
        o = attention(q, k, v, dev["q2k_idx"], dev["q2k_num"], dev["vbs"], case["sm_scale"],
                      k2q=given)
        o.backward(dev["do"])
        grads.append((o.detach(), q.grad, k.grad, v.grad))
    torch.cuda.synchronize()
    (o1, dq1, dk1, dv1), (o2, dq2, dk2, dv2) = grads
    assert torch.equal(o1, o2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dq1.float() - dq2.float()).abs().max() <= 5e-3 * dq1.float().abs().max()
