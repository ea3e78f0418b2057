"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle on the same seeded
inputs.

- inversion: bit-exact (counts, ids and the zero padding) on every workload and on random
  selections with invalid entries;
- backward and forward: the oracle's float64 result rounded to bf16, per tensor
  max|d| <= 1e-2 max|ref| and mean|d| <= 1e-3 mean|ref| (tests/parity.py), on small cases that
  span several work items, odd pair tails, ragged and empty blocks, unselected kv blocks and
  empty query rows; exact +0.0 for unselected kv blocks and padded kv rows;
- the full-size workloads, in the launch configuration the benchmark times (GPU forward ->
  inversion -> backward), on sampled query blocks and kv blocks that the oracle computes one by
  one;
- two backward runs agree (dK, dV bitwise; dQ within 5e-3 of max|dQ|).
"""
import numpy as np
import pytest
import torch

from block_sparse_video_tok_gb300 import workloads as wl
from oracle import oracle as orc
from tests.parity import (bf16_round, check_close, f64, oracle_backward, oracle_forward,
                          to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vsa():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from block_sparse_video_tok_gb300 import build
    build.build()
    from block_sparse_video_tok_gb300 import vsa as binding
    return binding


def zero_bits(t):
    return (t.view(torch.int16) == 0)


# ------------------------------------------------------------------------------ inversion


@pytest.mark.parametrize("name", list(wl.CONFIGS))
def test_invert_bit_exact_on_workloads(vsa, name):
    case = wl.make_config(name)
    nb = case["nb"]
    k_idx, k_num, bad = orc.invert(case["q2k_idx"], case["q2k_num"], nb)
    assert bad == 0
    dev = to_device(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g_idx, g_num = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], nb, dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(g_num.cpu().numpy(), k_num)
    assert np.array_equal(g_idx.cpu().numpy(), k_idx)
    assert int(err.item()) == 0


@pytest.mark.parametrize("H,nb,topk", [(2, 8192, 16), (8, 4096, 16), (2, 2048, 256),
                                        (2, 333, 100)])
def test_invert_bit_exact_long(vsa, H, nb, topk):
    """Long sequences, where the inversion's column slices are wider than 32 kv blocks, and an
    odd nb.  (The oracle's plain membership scan bounds nb * nb * topk here.)"""
    q2k_idx, q2k_num = wl.make_selection(1, H, nb, topk, seed=nb + topk)
    k_idx, k_num, bad = orc.invert(q2k_idx, q2k_num, nb)
    assert bad == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g_idx, g_num = vsa.vsa_invert_indices(torch.from_numpy(q2k_idx).cuda(),
                                          torch.from_numpy(q2k_num).cuda(), nb, dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(g_num.cpu().numpy(), k_num)
    assert np.array_equal(g_idx.cpu().numpy(), k_idx)
    assert int(err.item()) == 0


@pytest.mark.parametrize("seed", [0, 1])
def test_invert_invalid_entries(vsa, seed):
    rng = np.random.default_rng(seed)
    B, H, nb, topk = 2, 3, 37, 9
    idx = rng.integers(-3, nb + 3, size=(B, H, nb, topk)).astype(np.int32)
    num = rng.integers(-2, topk + 3, size=(B, H, nb)).astype(np.int32)
    k_idx, k_num, bad = orc.invert(idx, num, nb)
    assert bad > 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g_idx, g_num = vsa.vsa_invert_indices(torch.from_numpy(idx).cuda(),
                                          torch.from_numpy(num).cuda(), nb, dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(g_num.cpu().numpy(), k_num)
    assert np.array_equal(g_idx.cpu().numpy(), k_idx)
    assert int(err.item()) & (vsa.DEVERR_Q2K_ID | vsa.DEVERR_Q2K_COUNT) == (
        vsa.DEVERR_Q2K_ID | vsa.DEVERR_Q2K_COUNT)


# ------------------------------------------------------------------------------ small cases

SMALL_CASES = {
    "tiny": lambda: wl.make_config("tiny"),
    "base_nb8_topk4": lambda: wl.make_case(1, 4, 8, 4, seed=1),
    "batch2": lambda: wl.make_case(2, 2, 8, 4, seed=2),
    "ragged": lambda: wl.make_case(1, 2, 8, 4, vbs="ragged32", seed=3),
    "topk1": lambda: wl.make_case(1, 2, 8, 1, vbs="ragged32", seed=4),
    "topk2": lambda: wl.make_case(1, 2, 8, 2, vbs="ragged32", seed=5),
    "topk3": lambda: wl.make_case(1, 2, 8, 3, vbs="ragged32", seed=6),
    "topk5": lambda: wl.make_case(1, 2, 8, 5, vbs="ragged32", seed=7),
    "topk7": lambda: wl.make_case(1, 2, 8, 7, vbs="ragged32", seed=8),
    "nb1": lambda: wl.make_case(1, 3, 1, 1, seed=9),
    "nb3_odd": lambda: wl.make_case(1, 2, 3, 2, vbs="ragged32", seed=10),
    "nb16": lambda: wl.make_case(1, 2, 16, 3, vbs="ragged32", seed=11),
    "nb33_many_items": lambda: wl.make_case(2, 3, 33, 6, vbs="ragged32", seed=12),
    "zero_count_kv": lambda: wl.make_case(1, 2, 8, 4, vbs="ragged32", seed=13, kv_pool=[0, 1, 3,
                                                                                       4, 6, 7]),
    "4k_25pct": lambda: wl.make_config("4k_25pct"),
}


def _special(name, case):
    """Cases with hand-made structure on top of a drawn one."""
    if name == "zero_vbs_and_empty_rows":
        case["vbs"][2] = 0
        case["q2k_num"][0, 0, 1] = 0      # q block 1 selects nothing: O = 0, lse = -inf
        case["q2k_idx"][0, 1, 3, :] = 2   # q block 3 of head 1 selects only the empty block
    return case


SMALL_CASES["zero_vbs_and_empty_rows"] = lambda: _special(
    "zero_vbs_and_empty_rows", wl.make_case(1, 2, 6, 3, seed=14))


def _scaled_kv_blocks(case, factor):
    """K of kv block j multiplied by factor(j) (then rounded to bf16 again): with growing
    factors each block's scores exceed the previous maximum by several log2 units, so the online
    softmax of the forward moves its reference maximum and rescales O many times; with shrinking
    factors the first block holds the maximum and later P values are tiny."""
    k = case["k"].float()
    for j in range(case["nb"]):
        k[:, :, 64 * j:64 * (j + 1)] *= factor(j)
    case["k"] = k.to(torch.bfloat16)
    return case


# 128-token blocks (each a pair of 64-token tiles with one selection).
SMALL_CASES["blk128"] = lambda: wl.make_case(1, 2, 4, 2, vbs="ragged65", seed=31, blk=128)
SMALL_CASES["blk128_odd_nb_topk3"] = lambda: wl.make_case(1, 2, 5, 3, vbs="ragged40", seed=32,
                                                         blk=128)
SMALL_CASES["blk128_batch2_zero_kv"] = lambda: wl.make_case(2, 2, 6, 2, vbs="ragged65", seed=33,
                                                           kv_pool=[0, 2, 3, 5], blk=128)

# The backward hands out the last items of its grid in parts (shares of an item's step list).
# With 16 heads of 16 kv blocks the last 16 items are split; with 3 q blocks per row most items
# have two steps, so some parts have none, and kv blocks 14 and 15 (selected by no q block) give
# split items without any step.
SMALL_CASES["split_parts_short_lists"] = lambda: wl.make_case(1, 16, 16, 3, vbs="ragged32", seed=41,
                                                             kv_pool=list(range(14)))

SMALL_CASES["growing_scores"] = lambda: _scaled_kv_blocks(
    wl.make_case(1, 2, 16, 8, vbs="ragged32", seed=15), lambda j: 1.0 + j)
SMALL_CASES["shrinking_scores"] = lambda: _scaled_kv_blocks(
    wl.make_case(1, 2, 16, 8, vbs="ragged32", seed=16), lambda j: 16.0 - j)


def _run_small(vsa, case):
    B, H, S, nb = case["B"], case["H"], case["S"], case["nb"]
    o64, lse64 = oracle_forward(case)
    o_b = bf16_round(o64)
    lse32 = lse64.astype(np.float32)
    dq64, dk64, dv64 = oracle_backward(case, f64(o_b), lse32.astype(np.float64))
    dev = to_device(case)
    k2q_idx, k2q_num = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], nb)
    ws = torch.empty(vsa.vsa_bwd_workspace_bytes(B, H, S), dtype=torch.uint8, device="cuda")
    dq, dk, dv = vsa.vsa_bwd(dev["do"], dev["q"], dev["k"], dev["v"], o_b.cuda(),
                             torch.from_numpy(lse32).cuda(), k2q_idx, k2q_num, dev["vbs"],
                             case["sm_scale"], workspace=ws)
    assert vsa.vsa_read_device_error(ws) == 0
    return (o64, lse64), (dq64, dk64, dv64), (dq, dk, dv), k2q_num.cpu().numpy()


@pytest.mark.parametrize("name", list(SMALL_CASES))
def test_backward_matches_oracle(vsa, name):
    case = SMALL_CASES[name]()
    _, (dq64, dk64, dv64), (dq, dk, dv), k2q_num = _run_small(vsa, case)
    check_close("dq", dq, dq64)
    check_close("dk", dk, dk64)
    check_close("dv", dv, dv64)
    # Exact +0.0 for unselected kv blocks and padded kv rows.
    blk = case.get("blk", 64)
    vbs = np.clip(case["vbs"], 0, blk)
    for b in range(case["B"]):
        for h in range(case["H"]):
            for j in range(case["nb"]):
                lo = blk * j + (0 if k2q_num[b, h, j] == 0 else int(vbs[j]))
                rows = slice(lo, blk * (j + 1))
                assert zero_bits(dk[b, h, rows]).all() and zero_bits(dv[b, h, rows]).all(), (b, h, j)


def test_split_parts_are_reproducible(vsa):
    """Split items add their parts in a fixed order: two runs give the same dK and dV bits."""
    case = SMALL_CASES["split_parts_short_lists"]()
    _, _, (dq1, dk1, dv1), _ = _run_small(vsa, case)
    _, _, (dq2, dk2, dv2), _ = _run_small(vsa, case)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dq1.float() - dq2.float()).abs().max() <= 5e-3 * dq1.float().abs().max()


@pytest.mark.parametrize("name", list(SMALL_CASES))
def test_forward_matches_oracle(vsa, name):
    case = SMALL_CASES[name]()
    o64, lse64 = oracle_forward(case)
    dev = to_device(case)
    o, lse = vsa.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["q2k_idx"], dev["q2k_num"], dev["vbs"],
                         case["sm_scale"])
    torch.cuda.synchronize()
    check_close("o", o, o64)
    g = lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(lse64)
    assert np.array_equal(np.isneginf(g), empty)
    assert np.abs(g[~empty] - lse64[~empty]).max() <= 1e-4 * max(1.0, np.abs(lse64[~empty]).max())
    assert (o.view(torch.int16)[torch.from_numpy(empty).cuda()] == 0).all()


def test_device_error_bits_and_clean_results(vsa):
    """Out-of-range ids and counts are skipped/clamped and reported; the result equals that of
    the cleaned selection."""
    case = wl.make_case(1, 2, 8, 3, vbs="ragged32", seed=21)
    dirty = dict(case)
    idx = np.concatenate([case["q2k_idx"], np.full_like(case["q2k_idx"][..., :1], 99)], -1)
    dirty["q2k_idx"] = idx
    dirty["q2k_num"] = case["q2k_num"] + 1       # the extra slot (id 99) is active
    dirty["q2k_num"][0, 1, 2] = 17               # count past the row width
    dirty["vbs"] = case["vbs"].copy()
    clean_num = case["q2k_num"].copy()
    clean_idx = np.concatenate([case["q2k_idx"], np.full_like(case["q2k_idx"][..., :1], 0)], -1)
    clean_idx[0, 1, 2, 3] = clean_idx[0, 1, 2, 0]  # clamped count 4 reads the duplicate slot 0
    clean_num[0, 1, 2] = 4
    dev_d = to_device(dirty)
    ws = torch.empty(vsa.vsa_fwd_workspace_bytes(1, 2, 512), dtype=torch.uint8, device="cuda")
    o_d, lse_d = vsa.vsa_fwd(dev_d["q"], dev_d["k"], dev_d["v"], dev_d["q2k_idx"],
                             dev_d["q2k_num"], dev_d["vbs"], case["sm_scale"], workspace=ws)
    bits = vsa.vsa_read_device_error(ws)
    assert bits & vsa.DEVERR_Q2K_ID and bits & vsa.DEVERR_Q2K_COUNT
    clean = dict(case, q2k_idx=clean_idx, q2k_num=clean_num)
    dev_c = to_device(clean)
    o_c, lse_c = vsa.vsa_fwd(dev_c["q"], dev_c["k"], dev_c["v"], dev_c["q2k_idx"],
                             dev_c["q2k_num"], dev_c["vbs"], case["sm_scale"])
    torch.cuda.synchronize()
    assert torch.equal(o_d, o_c) and torch.equal(lse_d, lse_c)


# ------------------------------------------------------------------------------ full size


def _head_case(case, b, h):
    sub = {n: case[n][b:b + 1, h:h + 1].contiguous() for n in ("q", "k", "v", "do")}
    sub["q2k_idx"] = case["q2k_idx"][b:b + 1, h:h + 1]
    sub["q2k_num"] = case["q2k_num"][b:b + 1, h:h + 1]
    sub["vbs"] = case["vbs"]
    sub["sm_scale"] = case["sm_scale"]
    sub["blk"] = case.get("blk", 64)
    return sub


def _full_size(vsa, name, n_heads=2, n_q=3, n_kv=2, seed=0):
    case = wl.make_config(name)
    B, H, S, nb = case["B"], case["H"], case["S"], case["nb"]
    dev = to_device(case)
    o, lse = vsa.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["q2k_idx"], dev["q2k_num"], dev["vbs"],
                         case["sm_scale"])
    k2q_idx, k2q_num = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], nb)
    ws = torch.empty(vsa.vsa_bwd_workspace_bytes(B, H, S), dtype=torch.uint8, device="cuda")
    dq, dk, dv = vsa.vsa_bwd(dev["do"], dev["q"], dev["k"], dev["v"], o, lse, k2q_idx, k2q_num,
                             dev["vbs"], case["sm_scale"], workspace=ws)
    assert vsa.vsa_read_device_error(ws) == 0
    counts = k2q_num.cpu().numpy()
    rng = np.random.default_rng(seed)
    heads = [(int(rng.integers(B)), int(rng.integers(H))) for _ in range(n_heads)]
    results = []
    for b, h in heads:
        sub = _head_case(case, b, h)
        cnt = counts[b, h]
        q_s = sorted(set(int(x) for x in rng.choice(nb, n_q, replace=False)))
        # kv blocks with a moderate list length (the oracle recomputes every selecting row),
        # plus one no q block selects, when there is one.
        mid = np.flatnonzero((cnt > 0) & (cnt <= max(160, int(np.median(cnt)))))
        kv_s = sorted(set(int(x) for x in rng.choice(mid, n_kv, replace=False)))
        zero = np.flatnonzero(cnt == 0)
        kv_all = kv_s + ([int(zero[0])] if zero.size else [])
        sel = sub["q2k_idx"][0, 0]
        need = set(q_s)
        for j in kv_s:
            need.update(int(i) for i in range(nb) if j in sel[i, :sub["q2k_num"][0, 0, i]])
        need = sorted(need)
        o64, lse64 = oracle_forward(sub, qblocks=need)
        o_b = bf16_round(np.nan_to_num(o64))
        lse32 = lse64.astype(np.float32)
        dq64, dk64, dv64 = oracle_backward(sub, f64(o_b), np.nan_to_num(lse32.astype(np.float64)),
                                           qblocks=q_s, kvblocks=kv_all)
        blk = case.get("blk", 64)
        for i in q_s:
            r = slice(blk * i, blk * (i + 1))
            results.append(check_close("%s o[%d,%d,q%d]" % (name, b, h, i), o[b, h, r],
                                       o64[0, 0, r]))
            g = lse[b, h, r].cpu().numpy().astype(np.float64)
            assert np.abs(g - lse64[0, 0, r]).max() <= 1e-4 * max(1.0, np.abs(lse64[0, 0, r]).max())
            results.append(check_close("%s dq[%d,%d,q%d]" % (name, b, h, i), dq[b, h, r],
                                       dq64[0, 0, r]))
        for j in kv_all:
            r = slice(blk * j, blk * (j + 1))
            if cnt[j] == 0:
                assert zero_bits(dk[b, h, r]).all() and zero_bits(dv[b, h, r]).all()
                continue
            results.append(check_close("%s dk[%d,%d,kv%d]" % (name, b, h, j), dk[b, h, r],
                                       dk64[0, 0, r]))
            results.append(check_close("%s dv[%d,%d,kv%d]" % (name, b, h, j), dv[b, h, r],
                                       dv64[0, 0, r]))
    return dev, case, (o, lse, k2q_idx, k2q_num), (dq, dk, dv)


@pytest.mark.parametrize("name", ["32k_25pct", "65k_12pct_zipf", "video_dit_21x30x52",
                                  "32k_25pct_blk128"])
def test_full_size_sampled(vsa, name):
    _full_size(vsa, name)


def test_long_sequence_sampled(vsa):
    """524,288 tokens (8192 kv blocks, so the work order is sorted) at low density: sampled
    parity of O, lse, dQ, dK and dV, and exact zeros for unselected kv blocks."""
    _full_size(vsa, "524k_sparse")


def test_two_runs_agree_at_65k(vsa):
    dev, case, (o, lse, k2q_idx, k2q_num), (dq, dk, dv) = _full_size(vsa, "65k_12pct_zipf",
                                                                   n_heads=1, n_q=1, n_kv=1)
    dq2, dk2, dv2 = vsa.vsa_bwd(dev["do"], dev["q"], dev["k"], dev["v"], o, lse, k2q_idx, k2q_num,
                                dev["vbs"], case["sm_scale"])
    torch.cuda.synchronize()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    d = (dq.float() - dq2.float()).abs()
    assert d.max().item() <= 5e-3 * dq.float().abs().max().item()
