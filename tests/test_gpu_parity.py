"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle on the same seeded
inputs.

- inversion: bit-exact (counts, ids and the zero padding) on every workload and on random
  selections with invalid entries;
- backward and forward: the oracle's float64 result rounded to bf16, per tensor
  max|d| <= 1e-2 max|ref| and mean|d| <= 1e-3 mean|ref| (tests/parity.py), on small cases that
  span several work items, odd pair tails, ragged and empty blocks, unselected kv blocks and
  empty query rows; exact +0.0 for unselected kv blocks and padded kv rows;
- k2q ids outside [0, nb) are skipped and reported;
- the work order is bit-exact against the oracle's.
The full-size workloads are in test_gpu_full_size.py.
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

# The backward hands out the last items of its grid in parts (shares of an item's step list:
# halves with fewer than 8 items per SM, as in these cases, quarters otherwise).  With 16 heads
# of 16 kv blocks the last 32 items are split; with 3 q blocks per row most items have two
# steps, so some parts have one and some none, and kv blocks 14 and 15 (selected by no q block)
# give split items without any step.
SMALL_CASES["split_parts_short_lists"] = lambda: wl.make_case(1, 16, 16, 3, vbs="ragged32", seed=41,
                                                             kv_pool=list(range(14)))
# 4 heads of 64 kv blocks, 40 selected per q block: the 32 split items (the shortest lists of the
# last head, last in the sorted order) have 14 to 20 steps, 7 to 10 per part.
SMALL_CASES["split_parts_long_lists"] = lambda: wl.make_case(1, 4, 64, 40, vbs="ragged33", seed=42)

def _outliers(case, which="qkvd", factor=1e3, seed=0):
    """One element per (b, h) head of each named tensor (q, k, v, d = dO) replaced by
    +-3 * factor: about `factor` times the largest of the head's other N(0, 1) values.  Such an
    outlier sets the per-head scale of its tensor, which moves every other value of the head
    `log2(factor)` binades down the fp16 range of the kernels' operand copies."""
    rng = np.random.default_rng(seed)
    names = {"q": "q", "k": "k", "v": "v", "d": "do"}
    for w in which:
        t = case[names[w]].float()
        B, H, S, D = t.shape
        for b in range(B):
            for h in range(H):
                t[b, h, int(rng.integers(S)), int(rng.integers(D))] = \
                    float(rng.choice([-3.0, 3.0])) * factor
        case[names[w]] = t.to(torch.bfloat16)
    return case


def _head_scaled(case, factor=1e-3):
    """Odd heads' Q, K, V and dO multiplied by `factor` (rounded to bf16 again): heads whose
    values differ by three orders of magnitude in one call."""
    for n in ("q", "k", "v", "do"):
        t = case[n].float()
        t[:, 1::2] *= factor
        case[n] = t.to(torch.bfloat16)
    return case


# Outliers (fp16 operand scaling): every tensor at once on the tiny and 4k workloads; V and dO
# (the operands of dP, whose product sets the range of dS) at 8k tokens and full density, where
# P is as small as at 32k tokens and 25 %.
SMALL_CASES["outliers_tiny"] = lambda: _outliers(wl.make_config("tiny"), seed=81)
SMALL_CASES["outliers_4k"] = lambda: _outliers(wl.make_config("4k_25pct"), seed=82)
SMALL_CASES["outliers_v_do_8k_dense"] = lambda: _outliers(
    wl.make_case(1, 2, 128, 128, seed=83), which="vd", seed=83)
SMALL_CASES["head_scales_4k"] = lambda: _head_scaled(wl.make_config("4k_25pct"))

def _zero_tiles(case):
    """Tiles of zeros: V of kv tile 1 and K of kv tile 3 in head 0, and all of dO in head 1 --
    the per-tile and per-head scale exponents of zero groups, and a dS bound of zero."""
    for n, sl in (("v", (0, 0, slice(64, 128))), ("k", (0, 0, slice(192, 256))),
                  ("do", (0, 1, slice(None)))):
        t = case[n].clone()
        t[sl] = 0
        case[n] = t
    return case


SMALL_CASES["zero_tiles"] = lambda: _zero_tiles(wl.make_case(1, 2, 8, 4, vbs="ragged32", seed=91))

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


# ------------------------------------------------------------------------------ invalid k2q ids


def _dirty_k2q(k2q_idx, k2q_num, nb, rng, aligned, heads=(0,)):
    """Copy of a k2q list with ids outside [0, nb) added to every row of the given (flat) heads.
    aligned: the bad ids go in as a pair at an even position, so every step keeps its pair of
    valid q blocks (the dK/dV accumulation order is unchanged); else one bad id at position 1
    (the pairing shifts).  Every row of a head gets the same number of extra slots, so the
    head's work order (by count) is unchanged, and the other heads -- among them the last one,
    whose last items the backward splits into parts -- are left alone."""
    idx, num = k2q_idx.copy(), k2q_num.copy()
    B, H, _, width = idx.shape
    extra = 2 if aligned else 1
    for flat in heads:
        b, h = divmod(flat, H)
        for j in range(nb):
            n = int(num[b, h, j])
            assert n + extra <= width
            row = idx[b, h, j, :n].tolist()
            pos = 2 * int(rng.integers(0, n // 2 + 1)) if aligned else min(1, n)
            bad = [-1 - int(rng.integers(0, 5)), nb + int(rng.integers(0, 5))][:extra]
            row[pos:pos] = bad
            idx[b, h, j, :n + extra] = row
            num[b, h, j] = n + extra
    return idx, num


@pytest.mark.parametrize("aligned", [True, False])
def test_invalid_k2q_ids_are_skipped(vsa, aligned):
    """A k2q id outside [0, nb) is skipped and reported: the result equals that of the clean
    list (dK, dV bitwise when the bad ids keep the step pairs), and matches the oracle."""
    case = wl.make_case(1, 2, 16, 6, vbs="ragged32", seed=51)
    B, H, S, nb = case["B"], case["H"], case["S"], case["nb"]
    (o64, lse64), (dq64, dk64, dv64), (dq, dk, dv), _ = _run_small(vsa, case)
    o_b = bf16_round(o64).cuda()
    lse = torch.from_numpy(lse64.astype(np.float32)).cuda()
    dev = to_device(case)
    k2q_idx, k2q_num = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], nb)
    rng = np.random.default_rng(7)
    d_idx, d_num = _dirty_k2q(k2q_idx.cpu().numpy(), k2q_num.cpu().numpy(), nb, rng, aligned)
    assert (d_num > k2q_num.cpu().numpy()).any()
    ws = torch.empty(vsa.vsa_bwd_workspace_bytes(B, H, S), dtype=torch.uint8, device="cuda")
    outs = [torch.full_like(dev["q"], float("nan")) for _ in range(3)]
    g = vsa.vsa_bwd(dev["do"], dev["q"], dev["k"], dev["v"], o_b, lse,
                    torch.from_numpy(d_idx).cuda(), torch.from_numpy(d_num).cuda(), dev["vbs"],
                    case["sm_scale"], dq=outs[0], dk=outs[1], dv=outs[2], workspace=ws)
    bits = vsa.vsa_read_device_error(ws)
    assert bits & vsa.DEVERR_K2Q_ID and not bits & vsa.DEVERR_TIMEOUT
    check_close("dq", g[0], dq64)
    check_close("dk", g[1], dk64)
    check_close("dv", g[2], dv64)
    if aligned:
        assert torch.equal(g[1], dk) and torch.equal(g[2], dv)


# ------------------------------------------------------------------------------ work order


@pytest.mark.parametrize("name", ["65k_12pct_zipf", "ties", "long_rows"])
def test_work_order_bit_exact(vsa, name):
    """The backward's item order (vsa_work_order; the backward's preprocess places its items with
    the same device code) against the oracle's stable descending sort, bit for bit."""
    if name == "65k_12pct_zipf":
        q2k_idx, q2k_num = wl.make_selection(1, 8, 1024, 128, select="zipf", seed=0)
        _, k_num, _ = orc.invert(q2k_idx, q2k_num, 1024)
        max_q = 1024
    elif name == "ties":   # few distinct counts, some out of range: long runs of ties
        rng = np.random.default_rng(3)
        k_num = rng.integers(-2, 7, size=(2, 3, 1500)).astype(np.int32)
        max_q = 4
    else:                  # a head too long for the shared-memory copy of its counts
        rng = np.random.default_rng(4)
        k_num = rng.integers(0, 300, size=(1, 1, 65536)).astype(np.int32)
        max_q = 256
    want = orc.work_order(k_num, max_q)
    got = vsa.vsa_work_order(torch.from_numpy(k_num).cuda(), max_q)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), want)


def test_nan_stays_in_its_head(vsa):
    """A NaN in one head's Q shows up in that head's gradients (nothing masks it), and the other
    head -- with its own operand scales and work items -- gives the results of the clean run."""
    case = wl.make_case(1, 2, 8, 4, vbs="ragged32", seed=92)
    B, H, S, nb = case["B"], case["H"], case["S"], case["nb"]
    o64, lse64 = oracle_forward(case)
    o_b = bf16_round(o64).cuda()
    lse = torch.from_numpy(lse64.astype(np.float32)).cuda()
    dev = to_device(case)
    k2q_idx, k2q_num = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], nb)
    args = (dev["do"], dev["q"], dev["k"], dev["v"], o_b, lse, k2q_idx, k2q_num, dev["vbs"],
            case["sm_scale"])
    clean = vsa.vsa_bwd(*args)
    q_nan = dev["q"].clone()
    q_nan[0, 0, 5, 3] = float("nan")
    dirty = vsa.vsa_bwd(args[0], q_nan, *args[2:])
    torch.cuda.synchronize()
    for name, c, d in zip(("dq", "dk", "dv"), clean, dirty):
        assert torch.isnan(d[0, 0].float()).any(), name
        assert torch.isfinite(d[0, 1].float()).all(), name
    assert torch.equal(clean[1][0, 1], dirty[1][0, 1]) and torch.equal(clean[2][0, 1], dirty[2][0, 1])
    dq_c, dq_d = clean[0][0, 1].float(), dirty[0][0, 1].float()
    assert (dq_c - dq_d).abs().max() <= 5e-3 * dq_c.abs().max()
