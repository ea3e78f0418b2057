"""Helpers of the GPU parity tests: run the oracle on a case, run the CUDA path through the C ABI,
and compare with the tolerance the benchmark spec fixes.

Tolerance (per tensor, against the oracle's float64 result rounded to bf16 with round-to-
nearest-even, since the library returns bf16):
    max|got - ref| <= 1e-2 * max|ref|      and      mean|got - ref| <= 1e-3 * mean|ref|.
Comparing against the unrounded float64 result instead could not pass the mean rule: bf16
output rounding alone costs about 1.4e-3 * mean|x| for Gaussian-like data.
"""
import numpy as np
import torch

from oracle import oracle as orc

REL_MAX = 1e-2
MEAN_REL = 1e-3


def bf16_round(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16)


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def errors(got, ref64):
    """(max|d|/max|ref|, mean|d|/mean|ref|) of a bf16 tensor against bf16(ref)."""
    g = f64(got)
    r = f64(bf16_round(ref64))
    d = np.abs(g - r)
    return (float(d.max() / max(np.abs(r).max(), 1e-30)),
            float(d.mean() / max(np.abs(r).mean(), 1e-30)))


def check_close(name, got, ref64, rel_max=REL_MAX, mean_rel=MEAN_REL):
    g = f64(got)
    assert np.isfinite(g).all(), name + ": non-finite values"
    rm, mr = errors(got, ref64)
    assert rm <= rel_max and mr <= mean_rel, (
        "%s: max|d|/max|ref| = %.3e (tol %.0e), mean|d|/mean|ref| = %.3e (tol %.0e)" %
        (name, rm, rel_max, mr, mean_rel))
    return rm, mr


def oracle_forward(case, qblocks=None):
    """Oracle O (float64) and lse for a workload case (dict from workloads.make_case)."""
    return orc.fwd(f64(case["q"]), f64(case["k"]), f64(case["v"]), case["q2k_idx"],
                   case["q2k_num"], case["vbs"], case["sm_scale"], blk=case.get("blk", 64),
                   qblocks=qblocks)


def oracle_backward(case, o_bf16_f64, lse, qblocks=None, kvblocks=None):
    return orc.bwd(f64(case["q"]), f64(case["k"]), f64(case["v"]), o_bf16_f64, f64(case["do"]),
                   lse, case["q2k_idx"], case["q2k_num"], case["vbs"], case["sm_scale"],
                   blk=case.get("blk", 64), qblocks=qblocks, kvblocks=kvblocks)


def to_device(case, dev="cuda"):
    out = {}
    for n in ("q", "k", "v", "do"):
        if n in case:
            out[n] = case[n].to(dev).contiguous()
    out["q2k_idx"] = torch.from_numpy(np.ascontiguousarray(case["q2k_idx"])).to(dev)
    out["q2k_num"] = torch.from_numpy(np.ascontiguousarray(case["q2k_num"])).to(dev)
    out["vbs"] = torch.from_numpy(np.ascontiguousarray(case["vbs"])).to(dev)
    return out


# ------------------------------------------------------------------------------ whole-tensor checks


def kv_row_masks(case, k2q_num):
    """[B, H, S] bool on k2q_num's device: the kv rows that take part in the backward (their
    block is selected by some q block and the row lies below the block's valid size)."""
    blk, S = case.get("blk", 64), case["S"]
    k2q_num = torch.as_tensor(k2q_num)
    dev = k2q_num.device
    sel = (k2q_num > 0).repeat_interleave(blk, dim=2)
    vbs = torch.from_numpy(np.clip(case["vbs"], 0, blk)).to(dev).repeat_interleave(blk)
    u = torch.arange(S, device=dev) % blk
    return sel & (u < vbs)[None, None, :]


def identity_tolerances(dv, dk, o, dout, q, sm_scale, live, n_acc=0):
    """Per-head, per-column tolerances of the identities
        sum_t dV_t = sum_r dO_r   and   sum_t dK_t = sm_scale sum_r (dO_r . (O*_r - O_r)) q_r
    (exact gradient; O* the exact forward output, O the bf16 O the backward is given), as 6
    standard deviations of sums of independent, zero-mean errors bounded per element by:
      - 2^-8 |x| for each dV or dK element (bf16 output rounding, at most 2^-9 relative, plus the
        kernel's own error, about 2e-4 relative in the small cases), taken at the rms of the
        column over the kv rows that take part;
      - 2^-8 |O_rd| for each element of the given O (2^-9 for its rounding, the rest for the
        forward's error), so the dK identity's term dO_r . (O*_r - O_r) has a standard deviation
        of at most 2^-8 sqrt(sum_d (dO_rd O_rd)^2 / 3) (uniform errors);
    plus, for dV, one error that is not independent between rows: the fp32 accumulator of an
    item's dV^T takes n_acc additions (one per 16 query rows of its list), and an accumulation
    that rounds toward zero loses up to 2^-23 of the running sum at each.  Every item adds its q
    rows in ascending order, so after k additions the running sums of all items together hold
    about the prefix sum_{r < R_k} dO_r of the rows; the losses add up to at most
    n_acc 2^-23 max_R |sum_{r < R} dO_r| per column (the same shrink leaves sum_t dK_t, which is
    about 0, alone).  On the GPU the shrink measured 2^-26 per addition on average.
    Returns (tol_dv, tol_dk), each [B, H, 128] float64."""
    n = live.sum(dim=2, keepdim=True).clamp(min=1).double()
    eps = 2.0 ** -8
    w = live[..., None].double()
    rms_dv = ((dv.double() ** 2 * w).sum(dim=2) / n).sqrt()
    rms_dk = ((dk.double() ** 2 * w).sum(dim=2) / n).sqrt()
    prefix = dout.double().cumsum(dim=2).abs().amax(dim=2)            # max_R |sum_{r<R} dO_r|
    tol_dv = 6 * eps * n.sqrt() * rms_dv + n_acc * 2.0 ** -23 * prefix
    row = eps * ((dout.double() * o.double()) ** 2).sum(dim=3).div(3.0).sqrt()   # [B, H, S]
    extra = sm_scale * ((row[..., None] * q.double()) ** 2).sum(dim=2).sqrt()
    tol_dk = 6 * (eps * n.sqrt() * rms_dk + extra)
    return tol_dv, tol_dk


def check_zero_rows_and_identities(case, k2q_num, q, dout, o, dk, dv, record=None):
    """On every head: dK and dV rows that take no part (unselected kv block, padded kv row) are
    exactly +0.0, and the two identities of ``identity_tolerances`` hold within their
    tolerances.  Needs every query row to see at least one key.  Tensors on any one device.
    `record` (a dict), if given, receives the worst ratios and the relative size of the dV
    identity's residual."""
    live = kv_row_masks(case, k2q_num)
    dead = ~live
    assert (dk.view(torch.int16)[dead] == 0).all(), "dK rows of unselected/padded kv rows"
    assert (dv.view(torch.int16)[dead] == 0).all(), "dV rows of unselected/padded kv rows"
    # Additions into an item's fp32 dV^T accumulator: one per 16 query rows of its longest list.
    n_acc = 4 * (case.get("blk", 64) // 64) * int(torch.as_tensor(k2q_num).max().item())
    tol_dv, tol_dk = identity_tolerances(dv, dk, o, dout, q, case["sm_scale"], live, n_acc)
    sum_do = dout.double().sum(dim=2)
    signed = dv.double().sum(dim=2) - sum_do
    r_dv = signed.abs()
    if record is not None:
        record["dv_ratio"] = (r_dv / tol_dv).max().item()
        record["dk_ratio"] = (dk.double().sum(dim=2).abs() / tol_dk).max().item()
        rel = signed / sum_do.abs().clamp(min=1e-30)
        record["dv_residual_over_sum_dO"] = (rel.median().item(), rel.min().item(),
                                             rel.max().item())
        record["n_acc"] = n_acc
    assert (r_dv <= tol_dv).all(), "sum dV != sum dO: worst residual/tolerance %.3f" % (
        (r_dv / tol_dv).max().item())
    r_dk = dk.double().sum(dim=2).abs()
    assert (r_dk <= tol_dk).all(), "sum dK != 0: worst residual/tolerance %.3f" % (
        (r_dk / tol_dk).max().item())
    return (r_dv / tol_dv).max().item(), (r_dk / tol_dk).max().item()
