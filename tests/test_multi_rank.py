"""World-size-2 host-side tests of the multi-rank path, on CPU with the gloo backend.

- Head sharding: two ranks each run the CPU oracle's forward and backward on their own (b, h)
  heads; gathered, the results equal one process computing all heads (no data-path collective
  is needed because heads are independent).
- The benchmark's barrier / max / sum helpers give the max and sum over ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from block_sparse_video_tok_gb300 import sharding
from block_sparse_video_tok_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _f64(t):
    return t.to(torch.float64).numpy()


def _oracle(case):
    from oracle import oracle as orc
    q, k, v, do = (_f64(case[n].contiguous()) for n in ("q", "k", "v", "do"))
    idx = np.ascontiguousarray(case["q2k_idx"])
    num = np.ascontiguousarray(case["q2k_num"])
    o, lse = orc.fwd(q, k, v, idx, num, case["vbs"], case["sm_scale"])
    dq, dk, dv = orc.bwd(q, k, v, o, do, lse, idx, num, case["vbs"], case["sm_scale"])
    return np.concatenate([o, dq, dk, dv], axis=-1)


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = wl.make_case(2, 3, 4, 2, vbs="ragged32", seed=5)
        sub = sharding.shard_case(case, rank, world)
        local = torch.from_numpy(_oracle(sub)[0])           # [heads_owned, S, 4*128]
        sizes = [sharding.head_range(6, r, world) for r in range(world)]
        parts = [torch.zeros((b - a,) + tuple(local.shape[1:]), dtype=local.dtype)
                 for a, b in sizes]
        dist.all_gather(parts, local)                         # verification only
        import bench
        dev = torch.device("cpu")
        mx = bench.reduce_max(dist, float(rank + 1), dev)
        sm = bench.reduce_sum(dist, float(rank + 1), dev)
        bench.barrier(dist, dev)
        if rank == 0:
            np.save(os.path.join(out_dir, "gathered.npy"), torch.cat(parts).numpy())
            np.save(os.path.join(out_dir, "reduced.npy"), np.array([mx, sm]))
    finally:
        dist.destroy_process_group()


def test_head_ranges_partition():
    for n in (1, 5, 6, 24):
        for world in (1, 2, 3, 8):
            ranges = [sharding.head_range(n, r, world) for r in range(world)]
            covered = [h for a, b in ranges for h in range(a, b)]
            assert covered == list(range(n))
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1


def test_two_ranks_shard_heads_and_reduce(tmp_path):
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a rank did not finish")
        assert p.exitcode == 0
    gathered = np.load(tmp_path / "gathered.npy")
    mx, sm = np.load(tmp_path / "reduced.npy")
    assert mx == 2.0 and sm == 3.0
    case = wl.make_case(2, 3, 4, 2, vbs="ragged32", seed=5)
    full = _oracle(case).reshape(6, *gathered.shape[1:])
    assert np.array_equal(gathered, full)
