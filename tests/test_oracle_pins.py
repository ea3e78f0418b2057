"""Pins of the CPU oracle against facts outside itself (no GPU needed).

- inversion: a hand-worked fixture (tests/golden/invert_tiny.json) and a brute-force
  membership check on random selections with duplicates and invalid ids;
- forward: dense float64 attention with the equivalent -inf block mask (tests/dense_ref.py),
  and, at full density with full blocks, torch's scaled_dot_product_attention;
- backward: torch.autograd of the dense masked attention, central finite differences of
  L = sum(O * dO), the invariants sum_t dK_t = 0 and sum_t dV_t = sum_r dO_r, exact-zero rows,
  and closed forms (one visible key; Q = 0; O = 0 handed to the backward).
"""
import json
import os

import numpy as np
import pytest
import torch

from tests.dense_ref import block_mask, dense_forward_backward, rel_err

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_case(rng, B, H, nb, topk, D=128, blk=64, ragged=False, zero_pool=None):
    S = nb * blk
    q, k, v, do = (rng.standard_normal((B, H, S, D)) for _ in range(4))
    pool = np.arange(nb) if zero_pool is None else np.array(
        [j for j in range(nb) if j not in zero_pool])
    idx = np.stack([np.sort(rng.permutation(pool)[:topk]) for _ in range(B * H * nb)])
    idx = idx.reshape(B, H, nb, topk).astype(np.int32)
    num = np.full((B, H, nb), topk, np.int32)
    vbs = (rng.integers(blk // 2, blk + 1, nb) if ragged else np.full(nb, blk)).astype(np.int32)
    return q, k, v, do, idx, num, vbs


# ----------------------------------------------------------------------------- inversion


def test_invert_golden_fixture(oracle):
    with open(os.path.join(HERE, "golden", "invert_tiny.json")) as f:
        data = json.load(f)
    for case in data["cases"]:
        k2q_idx, k2q_num, bad = oracle.invert(case["q2k_idx"], case["q2k_num"], case["nb"])
        assert k2q_idx.tolist() == case["k2q_idx"], case["note"]
        assert k2q_num.tolist() == case["k2q_num"], case["note"]
        assert bad == case["bad"], case["note"]


def brute_force_k2q(idx, num, nb):
    """Collect (q, kv) pairs from the q2k entries, then group them by kv and sort."""
    B, H, nq, topk = idx.shape
    rows = {}
    for b in range(B):
        for h in range(H):
            for i in range(nq):
                c = int(min(max(num[b, h, i], 0), topk))
                for s in range(c):
                    j = int(idx[b, h, i, s])
                    if 0 <= j < nb:
                        rows.setdefault((b, h, j), set()).add(i)
    return rows


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_invert_brute_force(oracle, seed):
    rng = np.random.default_rng(seed)
    B, H, nb, topk = 2, 3, 11, 5
    idx = rng.integers(-2, nb + 2, size=(B, H, nb, topk)).astype(np.int32)
    num = rng.integers(-1, topk + 2, size=(B, H, nb)).astype(np.int32)
    k2q_idx, k2q_num, bad = oracle.invert(idx, num, nb)
    expect = brute_force_k2q(idx, num, nb)
    n_bad = 0
    for b in range(B):
        for h in range(H):
            for i in range(nb):
                c = int(num[b, h, i])
                n_bad += int(c < 0 or c > topk)
                for s in range(min(max(c, 0), topk)):
                    n_bad += int(not 0 <= idx[b, h, i, s] < nb)
            for j in range(nb):
                want = sorted(expect.get((b, h, j), set()))
                n = int(k2q_num[b, h, j])
                assert k2q_idx[b, h, j, :n].tolist() == want
                assert (k2q_idx[b, h, j, n:] == 0).all()
    assert bad == n_bad > 0


# ----------------------------------------------------------------------------- forward


@pytest.mark.parametrize("ragged,blk", [(False, 64), (True, 64), (True, 128)])
def test_forward_matches_dense_masked(oracle, ragged, blk):
    rng = np.random.default_rng(10 + ragged + blk)
    q, k, v, do, idx, num, vbs = rand_case(rng, 1, 2, 4, 2, blk=blk, ragged=ragged)
    sc = 0.0883883476483184
    o, lse = oracle.fwd(q, k, v, idx, num, vbs, sc, blk=blk)
    o_ref, lse_ref, *_ = dense_forward_backward(q, k, v, do, block_mask(idx, num, vbs, blk), sc)
    assert rel_err(o, o_ref) < 1e-12
    assert np.abs(lse - lse_ref).max() < 1e-12


def test_forward_full_density_is_dense_attention(oracle):
    rng = np.random.default_rng(3)
    nb = 4
    q, k, v, do, idx, num, vbs = rand_case(rng, 1, 2, nb, nb)
    sc = 0.125
    o, _ = oracle.fwd(q, k, v, idx, num, vbs, sc)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), scale=sc).numpy()
    assert rel_err(o, ref) < 1e-12


def test_forward_closed_forms(oracle):
    rng = np.random.default_rng(4)
    nb, blk, D = 3, 64, 128
    q, k, v, do, idx, num, _ = rand_case(rng, 1, 1, nb, 1)
    # One visible key (block 0, size 1) for every query: P = 1, O = v_0, lse = z_0.
    idx[:] = 0
    vbs = np.array([1, 0, 0], np.int32)
    sc = 0.1
    o, lse = oracle.fwd(q, k, v, idx, num, vbs, sc)
    assert np.array_equal(o[0, 0], np.broadcast_to(v[0, 0, 0], o[0, 0].shape))
    z = q[0, 0] @ k[0, 0, 0] * sc * 1.4426950408889634
    assert np.abs(lse[0, 0] - z).max() < 1e-12
    # Q = 0: every visible key has the same score, P is uniform over the n visible keys.
    vbs = np.array([64, 7, 0], np.int32)
    idx = np.zeros((1, 1, nb, 2), np.int32)
    idx[..., 1] = 1
    num = np.full((1, 1, nb), 2, np.int32)
    o, lse = oracle.fwd(np.zeros_like(q), k, v, idx, num, vbs, sc)
    visible = np.concatenate([v[0, 0, :64], v[0, 0, 64:71]])
    assert rel_err(o[0, 0], np.broadcast_to(visible.mean(0), o[0, 0].shape)) < 1e-13
    assert np.abs(lse - np.log2(71)).max() < 1e-12


def test_forward_empty_rows(oracle):
    rng = np.random.default_rng(5)
    q, k, v, do, idx, num, vbs = rand_case(rng, 1, 1, 3, 2)
    num[0, 0, 1] = 0          # q block 1 selects nothing
    vbs[:] = [64, 64, 0]
    idx[0, 0, 2] = [2, 2]     # q block 2 selects only an empty block
    o, lse = oracle.fwd(q, k, v, idx, num, vbs, 0.1)
    for i in (1, 2):
        rows = slice(64 * i, 64 * (i + 1))
        assert (o[0, 0, rows] == 0).all() and np.isneginf(lse[0, 0, rows]).all()
    dq, dk, dv = oracle.bwd(q, k, v, o, do, lse, idx, num, vbs, 0.1)
    assert (dq[0, 0, 64:] == 0).all()


def test_set_semantics_and_invalid_entries(oracle):
    rng = np.random.default_rng(6)
    q, k, v, do, idx, num, vbs = rand_case(rng, 1, 1, 4, 2)
    clean = idx.copy()
    messy = np.concatenate([idx, idx[..., :1], np.full_like(idx[..., :1], 77)], axis=-1)
    messy_num = num + 1       # duplicate of slot 0 counts once; id 77 lies past the count
    o1, l1 = oracle.fwd(q, k, v, clean, num, vbs, 0.1)
    o2, l2 = oracle.fwd(q, k, v, messy, messy_num, vbs, 0.1)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    bad_num = num + 2         # now the out-of-range id 77 is active: skipped
    o3, l3 = oracle.fwd(q, k, v, messy, bad_num, vbs, 0.1)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


# ----------------------------------------------------------------------------- backward


@pytest.mark.parametrize("ragged,zero_pool,blk", [(False, None, 64), (True, None, 64),
                                                   (True, (1,), 64), (True, (2,), 128)])
def test_backward_matches_autograd(oracle, ragged, zero_pool, blk):
    rng = np.random.default_rng(20 + ragged + blk)
    q, k, v, do, idx, num, vbs = rand_case(rng, 1, 2, 4, 2, blk=blk, ragged=ragged,
                                           zero_pool=zero_pool)
    sc = 0.0883883476483184
    mask = block_mask(idx, num, vbs, blk)
    o_ref, lse_ref, dq_ref, dk_ref, dv_ref = dense_forward_backward(q, k, v, do, mask, sc)
    o, lse = oracle.fwd(q, k, v, idx, num, vbs, sc, blk=blk)
    dq, dk, dv = oracle.bwd(q, k, v, o, do, lse, idx, num, vbs, sc, blk=blk)
    assert rel_err(dq, dq_ref) < 1e-10
    assert rel_err(dk, dk_ref) < 1e-10
    assert rel_err(dv, dv_ref) < 1e-10


def test_backward_finite_differences(oracle):
    """Central differences of L = sum(O * dO) on a 2-block case."""
    rng = np.random.default_rng(30)
    q, k, v, do, idx, num, vbs = rand_case(rng, 1, 1, 2, 1, ragged=True)
    idx[0, 0, 1, 0] = 0       # both q blocks look at kv block 0; kv block 1 unselected
    sc = 0.0883883476483184
    o, lse = oracle.fwd(q, k, v, idx, num, vbs, sc)
    grads = dict(zip("qkv", oracle.bwd(q, k, v, o, do, lse, idx, num, vbs, sc)))
    h = 1e-5
    for name in "qkv":
        for _ in range(6):
            pos = tuple(int(rng.integers(0, n)) for n in q.shape)
            if name != "q":   # pick a visible key row of block 0
                pos = (0, 0, int(rng.integers(0, vbs[0])), pos[3])
            args = {"q": q, "k": k, "v": v}
            plus = {n: a.copy() for n, a in args.items()}
            minus = {n: a.copy() for n, a in args.items()}
            plus[name][pos] += h
            minus[name][pos] -= h
            lp = (oracle.fwd(plus["q"], plus["k"], plus["v"], idx, num, vbs, sc)[0] * do).sum()
            lm = (oracle.fwd(minus["q"], minus["k"], minus["v"], idx, num, vbs, sc)[0] * do).sum()
            fd = (lp - lm) / (2 * h)
            an = grads[name][pos]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, pos, fd, an)


def test_backward_invariants_and_zero_rows(oracle):
    rng = np.random.default_rng(40)
    B, H, nb = 2, 2, 6
    q, k, v, do, idx, num, vbs = rand_case(rng, B, H, nb, 3, ragged=True, zero_pool=(2, 4))
    sc = 0.0883883476483184
    o, lse = oracle.fwd(q, k, v, idx, num, vbs, sc)
    dq, dk, dv = oracle.bwd(q, k, v, o, do, lse, idx, num, vbs, sc)
    # Rows of P sum to 1: sum_t dV_t = sum_r dO_r.  Rows of dS sum to 0: sum_t dK_t = 0.
    assert rel_err(dv.sum(axis=2), do.sum(axis=2)) < 1e-11
    assert np.abs(dk.sum(axis=2)).max() < 1e-11 * np.abs(dk).max() * dk.shape[2]
    # Unselected kv blocks and padded kv rows are exactly zero.
    for j in range(nb):
        lo = 64 * j + (0 if j in (2, 4) else int(vbs[j]))
        assert (dk[:, :, lo:64 * (j + 1)] == 0).all() and (dv[:, :, lo:64 * (j + 1)] == 0).all()


def test_backward_closed_forms(oracle):
    rng = np.random.default_rng(50)
    q, k, v, do, idx, num, _ = rand_case(rng, 1, 1, 2, 1)
    sc = 0.1
    # One visible key: P = 1 and dS = 0, so dQ = dK = 0 and dV_key = sum_r dO_r.
    idx[:] = 0
    vbs = np.array([1, 0], np.int32)
    o, lse = oracle.fwd(q, k, v, idx, num, vbs, sc)
    dq, dk, dv = oracle.bwd(q, k, v, o, do, lse, idx, num, vbs, sc)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    assert rel_err(dv[0, 0, 0], do[0, 0].sum(0)) < 1e-13
    # O = 0 handed to the backward: Delta = 0, dS = P * (dO V^T), checked with matrix algebra.
    vbs = np.array([64, 64], np.int32)
    idx = np.array([[[[0, 1], [1, 0]]]], np.int32)
    num = np.array([[[2, 1]]], np.int32)
    o, lse = oracle.fwd(q, k, v, idx, num, vbs, sc)
    dq, dk, dv = oracle.bwd(q, k, v, np.zeros_like(o), do, lse, idx, num, vbs, sc)
    mask = block_mask(idx, num, vbs, 64).numpy()[0, 0]
    s = np.where(mask, q[0, 0] @ k[0, 0].T * sc, -np.inf)
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ds = p * (do[0, 0] @ v[0, 0].T)
    assert rel_err(dq[0, 0], ds @ k[0, 0] * sc) < 1e-11
    assert rel_err(dk[0, 0], ds.T @ q[0, 0] * sc) < 1e-11
    assert rel_err(dv[0, 0], p.T @ do[0, 0]) < 1e-11


def test_backward_subsets_match_full(oracle):
    """Computing only some dQ rows / dK-dV blocks gives the same values as the full run."""
    rng = np.random.default_rng(60)
    B, H, nb = 1, 2, 5
    q, k, v, do, idx, num, vbs = rand_case(rng, B, H, nb, 2, ragged=True)
    sc = 0.0883883476483184
    o, lse = oracle.fwd(q, k, v, idx, num, vbs, sc)
    o_sub, lse_sub = oracle.fwd(q, k, v, idx, num, vbs, sc, qblocks=[3, 7])
    assert np.array_equal(o_sub[0, 0, 192:256], o[0, 0, 192:256])
    assert np.array_equal(lse_sub[0, 1, 128:192], lse[0, 1, 128:192])
    dq, dk, dv = oracle.bwd(q, k, v, o, do, lse, idx, num, vbs, sc)
    dq2, dk2, dv2 = oracle.bwd(q, k, v, o, do, lse, idx, num, vbs, sc, qblocks=[6],
                               kvblocks=[1, 9])
    assert np.array_equal(dq2[0, 1, 64:128], dq[0, 1, 64:128])
    assert np.array_equal(dk2[0, 0, 64:128], dk[0, 0, 64:128])
    assert np.array_equal(dv2[0, 1, 256:320], dv[0, 1, 256:320])


# ----------------------------------------------------------------------------- work order


def test_work_order_golden_fixture(oracle):
    with open(os.path.join(HERE, "golden", "work_order_tiny.json")) as f:
        data = json.load(f)
    for case in data["cases"]:
        got = oracle.work_order(np.asarray(case["k2q_num"], np.int32), case["max_q"])
        assert got.tolist() == case["order"], case["note"]


@pytest.mark.parametrize("seed", [0, 1])
def test_work_order_properties(oracle, seed):
    """Within every head: a permutation of the head's items, clamped counts non-increasing, and
    equal counts in ascending block order -- properties that fix a stable descending sort."""
    rng = np.random.default_rng(seed)
    B, H, nb, max_q = 2, 3, 257, 40
    num = rng.integers(-3, max_q + 6, size=(B, H, nb)).astype(np.int32)
    num[0, 1, :] = 7                       # a head of equal counts keeps block order
    order = oracle.work_order(num, max_q)
    flat = np.clip(num.reshape(-1), 0, max_q)
    for bh in range(B * H):
        seg = order[bh * nb:(bh + 1) * nb]
        assert sorted(seg.tolist()) == list(range(bh * nb, (bh + 1) * nb))
        c = flat[seg]
        assert np.all(c[:-1] >= c[1:])
        tie = c[:-1] == c[1:]
        assert np.all(seg[:-1][tie] < seg[1:][tie])
    assert order[nb:2 * nb].tolist() == list(range(nb, 2 * nb))
