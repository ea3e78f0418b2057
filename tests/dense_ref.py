"""Dense float64 attention with an explicit block mask, in plain PyTorch CPU ops.

An independent formulation used to pin the oracle: the whole [S, S] score matrix is formed,
keys outside the selected blocks or past variable_block_sizes are set to -inf (FastVideo,
compare main...vsa_bwd_fix, tests/test_block_sparse_bwd_sm100a.py, reference()), softmax is
torch.softmax, and gradients come from torch.autograd of loss = sum(O * dO).
"""
import math

import numpy as np
import torch

LOG2E = 1.4426950408889634


def block_mask(q2k_idx, q2k_num, vbs, blk):
    """Boolean [B, H, S, S] visibility mask built from q2k (set semantics, invalid ids skipped,
    counts clamped to [0, topk]) and the per-block valid-token counts."""
    idx = np.asarray(q2k_idx)
    num = np.asarray(q2k_num)
    vbs = np.asarray(vbs)
    B, H, nq, topk = idx.shape
    nb = vbs.size
    S = nb * blk
    sel = np.zeros((B, H, nq, nb), bool)
    for b in range(B):
        for h in range(H):
            for i in range(nq):
                c = int(min(max(num[b, h, i], 0), topk))
                for s in range(c):
                    j = int(idx[b, h, i, s])
                    if 0 <= j < nb:
                        sel[b, h, i, j] = True
    key_ok = np.zeros(S, bool)
    for j in range(nb):
        key_ok[j * blk:j * blk + int(min(max(vbs[j], 0), blk))] = True
    m = np.repeat(np.repeat(sel, blk, axis=2), blk, axis=3) & key_ok[None, None, None, :]
    return torch.from_numpy(m)


def dense_forward_backward(q, k, v, do, mask, sm_scale):
    """Returns (O, lse in M form, dQ, dK, dV), all float64 numpy.  Rows with no visible key
    are given O = 0, lse = -inf and zero dQ (their softmax is undefined)."""
    q, k, v, do = (torch.as_tensor(np.asarray(t, dtype=np.float64)) for t in (q, k, v, do))
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    scores = (q @ k.transpose(-1, -2)) * sm_scale
    scores = scores.masked_fill(~mask, float("-inf"))
    empty = ~mask.any(dim=-1, keepdim=True)
    safe = scores.masked_fill(empty, 0.0)
    p = torch.softmax(safe, dim=-1).masked_fill(empty, 0.0)
    out = p @ v
    loss = (out * do).sum()
    dq, dk, dv = torch.autograd.grad(loss, (q, k, v))
    lse = torch.logsumexp(scores, dim=-1) * LOG2E
    return (out.detach().numpy(), lse.detach().numpy(), dq.numpy(), dk.numpy(), dv.numpy())


def rel_err(got, ref):
    got, ref = np.asarray(got), np.asarray(ref)
    scale = max(np.abs(ref).max(), 1e-300)
    return float(np.abs(got - ref).max() / scale)


def default_scale(d):
    return 1.0 / math.sqrt(d)
