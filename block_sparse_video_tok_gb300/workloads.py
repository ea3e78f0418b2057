"""Seeded synthetic workloads for 64-token block-sparse video attention.

This module only draws inputs: bf16 Q, K, V, dO ~ N(0, 1), a q2k block selection, and the
per-block valid-token counts (variable_block_sizes).  It holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle can take their inputs from it.

Random numbers come from numpy's PCG64 generator (stable across machines and versions); fp32
draws are rounded to bf16 with round-to-nearest-even by torch.  Draw order for a case: Q, K, V,
dO, then the selection, then ragged block sizes.

Selection patterns (all rows hold distinct kv block ids, sorted ascending, count = topk):
  uniform  each q block picks topk kv blocks uniformly at random (a random subset);
  zipf     per (b, h) a random permutation assigns popularity ranks; the least popular 5% of
           kv blocks get weight 0 (so about 5% of kv blocks are selected by no q block), the
           rest weight 1/rank; each q block draws topk blocks without replacement with those
           weights (Gumbel top-k), which makes k2q list lengths strongly skewed;
  scores   top-k of uniform random block scores (the video-DiT selection).
Block-size patterns: full (all 64), last40 (all 64, last block 40), ragged (uniform integers in
[lo, 64]), cubes (a latent video grid tiled into 4x4x4 cubes, clipped at the grid edges;
"cubes:TxHxW" names the grid, plain "cubes" is 21x30x52).
"""
import math

import numpy as np
import torch

BLOCK = 64
HEAD_DIM = 128

# The five workloads, by what they are.
CONFIGS = {
    "tiny": dict(B=1, H=1, nb=8, topk=2, select="uniform", vbs="last40", seed=0),
    "4k_25pct": dict(B=1, H=8, nb=64, topk=16, select="uniform", vbs="full", seed=0),
    "32k_25pct": dict(B=1, H=8, nb=512, topk=128, select="uniform", vbs="full", seed=0),
    "65k_12pct_zipf": dict(B=1, H=8, nb=1024, topk=128, select="zipf", vbs="ragged33", seed=0),
    "video_dit_21x30x52": dict(B=2, H=12, nb=624, topk=78, select="scores", vbs="cubes",
                               seed=0),
}

# Long sequences at 25 % density (B=1, H=8, D=128), the shapes of the sm_100a kernel's published
# table beyond 65k tokens.  Benchmark workloads only: their inputs take several GB to draw.
LONG_CONFIGS = {
    "131k_25pct": dict(B=1, H=8, nb=2048, topk=512, select="uniform", vbs="full", seed=0),
    "262k_25pct": dict(B=1, H=8, nb=4096, topk=1024, select="uniform", vbs="full", seed=0),
    "524k_25pct": dict(B=1, H=8, nb=8192, topk=2048, select="uniform", vbs="full", seed=0),
    # 524k tokens at low density: long-sequence index arithmetic at a size the oracle can sample.
    "524k_sparse": dict(B=1, H=2, nb=8192, topk=16, select="uniform", vbs="ragged33", seed=0),
    # 32k tokens in 128-token blocks at 25 % density.
    "32k_25pct_blk128": dict(B=1, H=8, nb=256, topk=64, select="uniform", vbs="full", seed=0,
                             blk=128),
    # Wan2.1-1.3B-like layers (12 heads of 128): an 81-frame 480P latent (21 x 60 x 104) and a
    # 720P one (21 x 90 x 160) in 4x4x4 cubes, each q block attending to 12.5 % of the cubes.
    "wan480p_h12": dict(B=1, H=12, nb=2340, topk=293, select="scores", vbs="cubes:21x60x104",
                        seed=0),
    "wan720p_h12": dict(B=1, H=12, nb=5520, topk=690, select="scores", vbs="cubes:21x90x160",
                        seed=0),
}

VIDEO_GRID = (21, 30, 52)
VIDEO_CUBE = (4, 4, 4)


def video_cube_sizes(grid=VIDEO_GRID, cube=VIDEO_CUBE):
    """Valid tokens of each 4x4x4 cube of a (T, H, W) latent grid, cubes in t-major, h, w
    order; edge cubes are clipped to the grid."""
    counts = [math.ceil(g / c) for g, c in zip(grid, cube)]
    ext = []
    for g, c, n in zip(grid, cube, counts):
        ext.append([min(c, g - c * x) for x in range(n)])
    sizes = [a * b * d for a in ext[0] for b in ext[1] for d in ext[2]]
    return np.asarray(sizes, dtype=np.int32)


def _bf16(x32):
    return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16)


def _select(rng, kind, B, H, nb, topk, kv_pool=None):
    rows = B * H * nb
    if kind == "uniform":
        pool = np.arange(nb) if kv_pool is None else np.asarray(kv_pool)
        assert topk <= pool.size
        # The topk smallest of uniform keys per row; rows in chunks so the keys of long sequences
        # never sit in memory at once (the draws are the same as one (rows, pool) call).
        pick = np.empty((rows, topk), np.int64)
        chunk = max(1, (1 << 24) // pool.size)
        for r0 in range(0, rows, chunk):
            keys = rng.random((min(chunk, rows - r0), pool.size))
            part = np.argpartition(keys, topk - 1, axis=1)[:, :topk] if topk < pool.size else \
                np.argsort(keys, axis=1)
            pick[r0:r0 + keys.shape[0]] = pool[part]
    elif kind == "zipf":
        pick = np.empty((rows, topk), np.int64)
        n_zero = int(round(0.05 * nb))
        for bh in range(B * H):
            rank = rng.permutation(nb)  # rank[j] = popularity rank of kv block j (0 = most)
            logw = -np.log(rank + 1.0)
            logw[rank >= nb - n_zero] = -np.inf
            g = -np.log(-np.log(rng.random((nb, nb))))
            keys = logw[None, :] + g
            pick[bh * nb:(bh + 1) * nb] = np.argsort(-keys, axis=1, kind="stable")[:, :topk]
    elif kind == "scores":
        # The topk largest of uniform scores per row, in row chunks like "uniform".
        pick = np.empty((rows, topk), np.int64)
        chunk = max(1, (1 << 24) // nb)
        for r0 in range(0, rows, chunk):
            scores = rng.random((min(chunk, rows - r0), nb))
            pick[r0:r0 + scores.shape[0]] = (
                np.argpartition(-scores, topk - 1, axis=1)[:, :topk] if topk < nb else
                np.argsort(-scores, axis=1))
    else:
        raise ValueError(kind)
    pick = np.sort(pick, axis=1).astype(np.int32)
    return pick.reshape(B, H, nb, topk)


def _block_sizes(rng, kind, nb, blk=BLOCK):
    if kind == "full":
        return np.full(nb, blk, np.int32)
    if kind == "last40":
        v = np.full(nb, blk, np.int32)
        v[-1] = 40
        return v
    if kind.startswith("ragged"):
        lo = int(kind[len("ragged"):])
        return rng.integers(lo, blk + 1, size=nb).astype(np.int32)
    if kind.startswith("cubes"):
        grid = VIDEO_GRID if kind == "cubes" else tuple(int(x) for x in kind[6:].split("x"))
        v = video_cube_sizes(grid)
        assert v.size == nb, (v.size, nb)
        return v
    raise ValueError(kind)


def make_case(B, H, nb, topk, select="uniform", vbs="full", seed=0, kv_pool=None,
              with_grad_out=True, blk=BLOCK):
    """Draw one case with nb sparse blocks of `blk` tokens (64 or 128).  Returns a dict with bf16
    CPU tensors q, k, v, do ([B,H,S,128], S = blk * nb), int32 numpy arrays q2k_idx
    [B,H,nb,topk], q2k_num [B,H,nb], vbs [nb], sm_scale and blk."""
    rng = np.random.Generator(np.random.PCG64(seed))
    S = nb * blk
    shape = (B, H, S, HEAD_DIM)
    names = ["q", "k", "v"] + (["do"] if with_grad_out else [])
    case = {}
    for n in names:
        case[n] = _bf16(rng.standard_normal(shape, dtype=np.float32))
    case["q2k_idx"] = _select(rng, select, B, H, nb, topk, kv_pool)
    case["q2k_num"] = np.full((B, H, nb), topk, np.int32)
    case["vbs"] = _block_sizes(rng, vbs, nb, blk)
    case["sm_scale"] = 1.0 / math.sqrt(HEAD_DIM)
    case.update(B=B, H=H, S=S, nb=nb, topk=topk, blk=blk)
    return case


def make_selection(B, H, nb, topk, select="uniform", seed=0):
    """Only a q2k selection (int32 [B,H,nb,topk], counts all topk), from its own generator."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return _select(rng, select, B, H, nb, topk), np.full((B, H, nb), topk, np.int32)


def make_config(name, seed=None):
    cfg = dict(CONFIGS[name] if name in CONFIGS else LONG_CONFIGS[name])
    if seed is not None:
        cfg["seed"] = seed
    return make_case(cfg["B"], cfg["H"], cfg["nb"], cfg["topk"], cfg["select"], cfg["vbs"],
                     cfg["seed"], blk=cfg.get("blk", BLOCK))


def selected_pairs(q2k_idx, q2k_num, nb):
    """Number of distinct (q block, kv block) pairs a selection names (ids in range only)."""
    idx = np.asarray(q2k_idx)
    num = np.asarray(q2k_num)
    B, H, nq, topk = idx.shape
    total = 0
    flat_idx = idx.reshape(-1, topk)
    flat_num = np.clip(num.reshape(-1), 0, topk)
    for r in range(flat_idx.shape[0]):
        row = flat_idx[r, :flat_num[r]]
        row = row[(row >= 0) & (row < nb)]
        total += np.unique(row).size
    return int(total)


def to_f64(t):
    """Exact widening of a bf16 tensor to a float64 numpy array."""
    return t.to(torch.float64).numpy()
