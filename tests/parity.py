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
