"""Python front end of the CPU oracle (``vsa_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the product package never does.  It builds the C oracle
with gcc on first use (into ``oracle/_build``) and exposes numpy-level wrappers.  All floating
point inputs are converted to float64; index inputs to int32.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libvsa_oracle.so")
_lib = None


def build(force=False):
    """Compile the oracle shared library (gcc, OpenMP).  Returns its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_variant(source_text, tag):
    """Compile an alternative oracle source (used by the tests that plant a mistake in a copy
    of the oracle to show the pins catch it).  Returns a loaded ctypes library."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_BUILD, "variant_%s.c" % tag)
    lib = os.path.join(_BUILD, "variant_%s.%d.so" % (tag, os.getpid()))
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", lib, src, "-lm"])
    handle = _declare(ctypes.CDLL(lib))
    os.remove(lib)  # the loaded image stays mapped
    os.remove(src)
    return handle


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_long
_D = ctypes.c_double


def _declare(lib):
    lib.vsa_oracle_num_threads.restype = _I
    lib.vsa_oracle_invert.restype = _L
    lib.vsa_oracle_invert.argtypes = [_P, _P, _I, _I, _I, _I, _I, _P, _P]
    lib.vsa_oracle_fwd.restype = _L
    lib.vsa_oracle_fwd.argtypes = [_P, _P, _P, _P, _P, _I, _P, _D, _I, _I, _I, _I, _I, _P, _L,
                                   _P, _P]
    lib.vsa_oracle_bwd.restype = _L
    lib.vsa_oracle_bwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _D, _I, _I, _I, _I,
                                   _I, _P, _L, _P, _L, _P, _P, _P]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def num_threads(lib=None):
    return (lib or _load()).vsa_oracle_num_threads()


def invert(q2k_idx, q2k_num, nb, lib=None):
    """q2k_idx [B,H,Nq,topk], q2k_num [B,H,Nq] -> (k2q_idx [B,H,nb,Nq], k2q_num [B,H,nb],
    number of invalid q2k entries)."""
    lib = lib or _load()
    idx, num = _i32(q2k_idx), _i32(q2k_num)
    B, H, nq, topk = idx.shape
    k2q_idx = np.empty((B, H, nb, nq), np.int32)
    k2q_num = np.empty((B, H, nb), np.int32)
    bad = lib.vsa_oracle_invert(_ptr(idx), _ptr(num), B, H, nq, topk, nb, _ptr(k2q_idx),
                                _ptr(k2q_num))
    return k2q_idx, k2q_num, bad


def fwd(q, k, v, q2k_idx, q2k_num, vbs, sm_scale, blk=64, qblocks=None, lib=None):
    """Block-sparse forward.  Returns (O [B,H,S,D], lse [B,H,S] in M form).  With ``qblocks``
    (flat ids bh*nq+i) only those query blocks are computed; the other rows are NaN."""
    lib = lib or _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    idx, num, vb = _i32(q2k_idx), _i32(q2k_num), _i32(vbs)
    B, H, S, D = q.shape
    o = np.full((B, H, S, D), np.nan)
    lse = np.full((B, H, S), np.nan)
    qb = None if qblocks is None else _i32(qblocks)
    n_qb = 0 if qb is None else qb.size
    lib.vsa_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(num), idx.shape[-1], _ptr(vb),
                       float(sm_scale), B, H, S, D, blk, _ptr(qb), n_qb, _ptr(o), _ptr(lse))
    return o, lse


def bwd(q, k, v, o, do, lse, q2k_idx, q2k_num, vbs, sm_scale, blk=64, qblocks=None,
        kvblocks=None, lib=None):
    """Block-sparse backward.  Returns (dQ, dK, dV) [B,H,S,D].  ``qblocks`` restricts the dQ
    rows computed, ``kvblocks`` the dK/dV rows (flat ids bh*nb+j); the rest are NaN."""
    lib = lib or _load()
    q, k, v, o, do, lse = (_f64(t) for t in (q, k, v, o, do, lse))
    idx, num, vb = _i32(q2k_idx), _i32(q2k_num), _i32(vbs)
    B, H, S, D = q.shape
    dq = np.full((B, H, S, D), np.nan)
    dk = np.full((B, H, S, D), np.nan)
    dv = np.full((B, H, S, D), np.nan)
    qb = None if qblocks is None else _i32(qblocks)
    kb = None if kvblocks is None else _i32(kvblocks)
    lib.vsa_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(idx),
                       _ptr(num), idx.shape[-1], _ptr(vb), float(sm_scale), B, H, S, D, blk,
                       _ptr(qb), 0 if qb is None else qb.size, _ptr(kb),
                       0 if kb is None else kb.size, _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv


def work_order(k2q_num, max_q):
    """The backward's work order: the FastVideo sm_100a backward's commit message (Semantics)
    sorts the (batch, head, kv block) items by the length of their k2q lists from 1024 kv blocks
    on, and its launch header (compare main...vsa_bwd_fix, ORDER_MIN_KV_BLOCKS) keeps the (b, h)
    segments in head order.  Plain definition: for each (b, h) in order, its kv blocks j by
    DESCENDING count (clamped to [0, max_q], the bounded active prefix of cudnn-frontend PR #926,
    Summary), equal counts in ascending j (a stable sort; Python's sort is stable).  Returns
    int32 [B * H * nb] of flat item ids bh * nb + j."""
    num = np.asarray(k2q_num).reshape(-1, np.asarray(k2q_num).shape[-1])
    n_heads, nb = num.shape
    out = []
    for bh in range(n_heads):
        counts = [min(max(int(c), 0), int(max_q)) for c in num[bh]]
        for j in sorted(range(nb), key=lambda x: -counts[x]):
            out.append(bh * nb + j)
    return np.asarray(out, dtype=np.int32)
