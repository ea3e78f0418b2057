"""Partition of block-sparse attention work over ranks by (batch, head).

Every work item, dQ row and dK/dV row of the backward belongs to one (b, h) head, so splitting
the B*H heads into contiguous ranges gives independent problems with no collective on the data
path.  These helpers are host-side index bookkeeping only.
"""


def head_range(num_heads, rank, world):
    """Contiguous [start, stop) of the flattened (b, h) heads owned by `rank`; the ranges cover
    0..num_heads-1 exactly once and their sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world: %d/%d" % (rank, world))
    base, extra = divmod(num_heads, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_case(case, rank, world):
    """The heads of `rank` as a case of their own (B = 1, H = heads owned), from a workload dict
    as drawn by workloads.make_case.  Activations are views of the flattened [B*H, S, 128]."""
    B, H = case["B"], case["H"]
    start, stop = head_range(B * H, rank, world)
    sub = dict(case)
    for n in ("q", "k", "v", "do"):
        if n in case:
            t = case[n]
            sub[n] = t.reshape(1, B * H, *t.shape[2:])[:, start:stop]
    for n in ("q2k_idx", "q2k_num"):
        a = case[n]
        sub[n] = a.reshape(1, B * H, *a.shape[2:])[:, start:stop]
    sub["B"], sub["H"] = 1, stop - start
    sub["heads"] = (start, stop)
    return sub
