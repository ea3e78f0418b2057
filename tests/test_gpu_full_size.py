"""Full-size parity: the five workloads' large members, the 128-token-block and long-sequence
workloads, run in the configuration the benchmark times (GPU forward -> inversion -> backward,
through the C ABI), with every output element accounted for.

- Outputs start as NaN, so an element the backward never writes shows up.
- Every head: all of dQ, dK, dV finite; every kv row of an unselected kv block and every padded
  kv row (at or past variable_block_sizes) exactly +0.0 in dK and dV; and two identities that
  hold for the exact gradient whatever the data (rows of P sum to one, rows of dS sum to zero):
      sum_t dV_t = sum_r dO_r,
      sum_t dK_t = sm_scale sum_r (dO_r . (O*_r - O_r)) q_r    (O* exact, O the bf16 O given),
  each within the tolerance worked out in tests/parity.py (``identity_tolerances``).
- One whole (b, h) head compared with the oracle element by element (forward O and lse; backward
  dQ, dK, dV).  It is the last head in claim order, which holds every item the backward splits
  into parts (the grid's last claims).  The kv block with the longest k2q list of the whole
  workload (the first item the sorted order hands out) is compared too.
- The work order the backward uses bit for bit against the oracle's.
The backward gets the GPU forward's O and lse; the oracle's backward is given the same O and lse,
and the GPU forward itself is checked against the oracle's forward on the whole head.
"""
import math

import numpy as np
import pytest
import torch

from block_sparse_video_tok_gb300 import workloads as wl
from oracle import oracle as orc
from tests.parity import (check_close, check_zero_rows_and_identities, f64, oracle_backward,
                          oracle_forward, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vsa():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from block_sparse_video_tok_gb300 import build
    build.build()
    from block_sparse_video_tok_gb300 import vsa as binding
    return binding


def head_case(case, b, h):
    sub = {n: case[n][b:b + 1, h:h + 1].contiguous() for n in ("q", "k", "v", "do")}
    sub["q2k_idx"] = case["q2k_idx"][b:b + 1, h:h + 1]
    sub["q2k_num"] = case["q2k_num"][b:b + 1, h:h + 1]
    sub["vbs"] = case["vbs"]
    sub["sm_scale"] = case["sm_scale"]
    sub["blk"] = case.get("blk", 64)
    return sub


def run_chain(vsa, case):
    """GPU forward -> inversion -> backward on NaN-filled outputs."""
    B, H, S, nb = case["B"], case["H"], case["S"], case["nb"]
    dev = to_device(case)
    o, lse = vsa.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["q2k_idx"], dev["q2k_num"], dev["vbs"],
                         case["sm_scale"])
    k2q_idx, k2q_num = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], nb)
    ws = torch.empty(vsa.vsa_bwd_workspace_bytes(B, H, S), dtype=torch.uint8, device="cuda")
    outs = [torch.full_like(dev["q"], float("nan")) for _ in range(3)]
    grads = vsa.vsa_bwd(dev["do"], dev["q"], dev["k"], dev["v"], o, lse, k2q_idx, k2q_num,
                        dev["vbs"], case["sm_scale"], dq=outs[0], dk=outs[1], dv=outs[2],
                        workspace=ws)
    assert vsa.vsa_read_device_error(ws) == 0
    return dev, (o, lse, k2q_idx, k2q_num), grads


def check_every_head(case, dev, fwd, grads):
    o, lse, _, k2q_num = fwd
    dq, dk, dv = grads
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv), ("o", o)):
        assert torch.isfinite(t).all(), name + ": non-finite (or never written) elements"
    # Every query row here sees at least one key (each q block selects blocks with rows), so
    # its P row sums to one and its dS row to zero.
    assert torch.isfinite(lse).all()
    rec = {}
    try:
        check_zero_rows_and_identities(case, k2q_num, dev["q"], dev["do"], o, dk, dv, rec)
    finally:
        print("identities %s: %s" % (case["S"], rec))


def check_whole_head(case, fwd, grads, b, h, label):
    o, lse, _, _ = fwd
    dq, dk, dv = grads
    sub = head_case(case, b, h)
    o64, lse64 = oracle_forward(sub)
    check_close("%s o[%d,%d]" % (label, b, h), o[b, h], o64[0, 0])
    g = lse[b, h].cpu().numpy().astype(np.float64)
    assert np.abs(g - lse64[0, 0]).max() <= 1e-4 * max(1.0, np.abs(lse64[0, 0]).max())
    o_in = f64(o[b:b + 1, h:h + 1])
    lse_in = f64(lse[b:b + 1, h:h + 1])
    dq64, dk64, dv64 = oracle_backward(sub, o_in, lse_in)
    check_close("%s dq[%d,%d]" % (label, b, h), dq[b, h], dq64[0, 0])
    check_close("%s dk[%d,%d]" % (label, b, h), dk[b, h], dk64[0, 0])
    check_close("%s dv[%d,%d]" % (label, b, h), dv[b, h], dv64[0, 0])


def check_blocks(case, fwd, grads, b, h, qblocks, kvblocks, label):
    """Sampled blocks of one head: O, lse and dQ of `qblocks`, dK and dV of `kvblocks`."""
    o, lse, _, _ = fwd
    dq, dk, dv = grads
    blk = case.get("blk", 64)
    sub = head_case(case, b, h)
    if qblocks:
        o64, lse64 = oracle_forward(sub, qblocks=qblocks)
        for i in qblocks:
            r = slice(blk * i, blk * (i + 1))
            check_close("%s o[%d,%d,q%d]" % (label, b, h, i), o[b, h, r], o64[0, 0, r])
            g = lse[b, h, r].cpu().numpy().astype(np.float64)
            assert np.abs(g - lse64[0, 0, r]).max() <= 1e-4 * max(1.0, np.abs(lse64[0, 0, r]).max())
    o_in = f64(o[b:b + 1, h:h + 1])
    lse_in = f64(lse[b:b + 1, h:h + 1])
    dq64, dk64, dv64 = oracle_backward(sub, o_in, lse_in, qblocks=list(qblocks),
                                       kvblocks=list(kvblocks))
    for i in qblocks:
        r = slice(blk * i, blk * (i + 1))
        check_close("%s dq[%d,%d,q%d]" % (label, b, h, i), dq[b, h, r], dq64[0, 0, r])
    for j in kvblocks:
        r = slice(blk * j, blk * (j + 1))
        check_close("%s dk[%d,%d,kv%d]" % (label, b, h, j), dk[b, h, r], dk64[0, 0, r])
        check_close("%s dv[%d,%d,kv%d]" % (label, b, h, j), dv[b, h, r], dv64[0, 0, r])


def check_work_order(vsa, case, k2q_num):
    """The backward takes its items in the order vsa_work_order computes (the same device code
    places them in the backward's preprocess); check it bit for bit against the oracle."""
    got = vsa.vsa_work_order(k2q_num, case["nb"], block=case.get("blk", 64))
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), orc.work_order(k2q_num.cpu().numpy(), case["nb"]))


def longest_list(k2q_num):
    flat = int(torch.argmax(k2q_num.reshape(-1)).item())
    B, H, nb = k2q_num.shape
    return flat // (H * nb), (flat // nb) % H, flat % nb


@pytest.mark.parametrize("name", ["32k_25pct", "65k_12pct_zipf", "video_dit_21x30x52",
                                  "32k_25pct_blk128"])
def test_full_size_whole_head(vsa, name):
    case = wl.make_config(name)
    B, H = case["B"], case["H"]
    dev, fwd, grads = run_chain(vsa, case)
    check_every_head(case, dev, fwd, grads)
    check_work_order(vsa, case, fwd[3])
    b, h = B - 1, H - 1
    check_whole_head(case, fwd, grads, b, h, name)
    lb, lh, lj = longest_list(fwd[3])
    if (lb, lh) != (b, h):
        check_blocks(case, fwd, grads, lb, lh, [], [lj], name + " longest")


@pytest.mark.parametrize("name", ["131k_25pct", "262k_25pct", "524k_25pct", "524k_sparse",
                                  "wan480p_h12"])
def test_long_sequence_sampled(vsa, name):
    """Sequences of 131,072, 262,144 and 524,288 tokens at 25 % density (2048, 4096 and 8192 kv
    blocks), 524,288 tokens at low density and a Wan 480P-like layer (12 heads, 149,760 tokens in
    2340 clipped 4x4x4 cubes, 12.5 %): every head as above; sampled q and kv blocks of the last
    head (including its shortest lists, the split items) and the longest list, against the
    oracle."""
    case = wl.make_config(name)
    B, H, nb = case["B"], case["H"], case["nb"]
    dev, fwd, grads = run_chain(vsa, case)
    check_every_head(case, dev, fwd, grads)
    check_work_order(vsa, case, fwd[3])
    counts = fwd[3][B - 1, H - 1].cpu().numpy()
    rng = np.random.default_rng(5)
    live = np.flatnonzero(counts > 0)
    order = live[np.argsort(counts[live], kind="stable")]
    kv = sorted({int(order[0]), int(order[1]), int(rng.choice(live))})   # two shortest, one any
    qs = sorted(int(x) for x in rng.choice(nb, 2, replace=False))
    check_blocks(case, fwd, grads, B - 1, H - 1, qs, kv, name)
    lb, lh, lj = longest_list(fwd[3])
    check_blocks(case, fwd, grads, lb, lh, [], [lj], name + " longest")


def test_two_runs_agree_at_65k(vsa):
    """dK and dV involve no atomics: bit-identical across runs; dQ's fp32 partial sums are added
    in a varying order: within 5e-3 of max|dQ| (the pages' run-to-run figure)."""
    case = wl.make_config("65k_12pct_zipf")
    dev, (o, lse, k2q_idx, k2q_num), (dq, dk, dv) = run_chain(vsa, case)
    dq2, dk2, dv2 = vsa.vsa_bwd(dev["do"], dev["q"], dev["k"], dev["v"], o, lse, k2q_idx, k2q_num,
                                dev["vbs"], case["sm_scale"])
    torch.cuda.synchronize()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    d = (dq.float() - dq2.float()).abs()
    assert d.max().item() <= 5e-3 * dq.float().abs().max().item()
    assert math.isfinite(d.max().item())
