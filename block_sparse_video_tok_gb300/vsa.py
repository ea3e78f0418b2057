"""Thin Python binding of libvsa.so (include/vsa.h), with the C entry points' names.

Argument marshalling only: shapes, dtypes and pointers of torch CUDA tensors are checked and
passed through ctypes; every step of the computation runs in the library's CUDA kernels.
Outputs and workspaces that the caller does not pass are allocated here with torch (the library
itself never allocates).  If libvsa.so has not been built this module raises on first use; there
is no fallback implementation.
"""
import ctypes
import os

import torch

from . import build as _build

BLOCK = 64
HEAD_DIM = 128

# Device error bits (include/vsa.h).
DEVERR_Q2K_ID = 0x01
DEVERR_Q2K_COUNT = 0x02
DEVERR_K2Q_ID = 0x04
DEVERR_K2Q_COUNT = 0x08
DEVERR_VBS = 0x10
DEVERR_TIMEOUT = 0x20


class VsaShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("seqlen", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block", ctypes.c_int32)]


class VsaBwdEvents(ctypes.Structure):
    _fields_ = [("start", ctypes.c_void_p), ("before_main", ctypes.c_void_p),
                ("after_main", ctypes.c_void_p), ("end", ctypes.c_void_p)]


class VsaError(RuntimeError):
    """A libvsa call returned a non-OK status."""


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_lib = None

# Every symbol include/vsa.h declares, with its (restype, argtypes).
SIGNATURES = {
    "vsa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "vsa_last_cuda_error": (ctypes.c_int, []),
    "vsa_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "vsa_invert_indices": (ctypes.c_int, [_P, _P, _I32, VsaShape, _P, _P, _P, _P]),
    "vsa_fwd_workspace_bytes": (_SZ, [VsaShape]),
    "vsa_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _P, _F, VsaShape, _P, _P, _P, _SZ, _P]),
    "vsa_bwd_workspace_bytes": (_SZ, [VsaShape]),
    "vsa_work_order": (ctypes.c_int, [_P, _I32, VsaShape, _P, _P]),
    "vsa_bwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _F, VsaShape, _P, _P,
                               _P, _P, _SZ, _P]),
    "vsa_bwd_timed": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _F, VsaShape, _P,
                                     _P, _P, _P, _SZ, ctypes.POINTER(VsaBwdEvents), _P]),
    "vsa_bwd_no_alloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _F, VsaShape,
                                        _P, _P, _P, _P]),
    "vsa_bwd_no_alloc_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), _P]),
    "vsa_read_device_error": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
}


def library_path():
    return _build.LIB


def lib():
    """The loaded libvsa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError("libvsa.so is not built (%s); build it with "
                               "block_sparse_video_tok_gb300.build.build()" % path)
        handle = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status):
    return lib().vsa_status_string(int(status)).decode()


def _check(status, what):
    if status != 0:
        raise VsaError("%s failed: %s (last CUDA error %d)" %
                       (what, status_string(status), lib().vsa_last_cuda_error()))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must be %d-D, got %s" % (name, ndim, tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def make_shape(batch, heads, seqlen, head_dim=HEAD_DIM, block=BLOCK):
    return VsaShape(int(batch), int(heads), int(seqlen), int(head_dim), int(block))


def _block_size(S, vbs):
    """Tokens per sparse block, inferred from the sequence length and the number of blocks (the
    length of variable_block_sizes): 64 or 128."""
    nb = vbs.numel()
    if nb < 1 or S % nb != 0 or S // nb not in (64, 128):
        raise ValueError("S = %d is not 64 or 128 tokens times len(vbs) = %d" % (S, nb))
    return S // nb


def vsa_fwd_workspace_bytes(batch, heads, seqlen, head_dim=HEAD_DIM):
    return int(lib().vsa_fwd_workspace_bytes(make_shape(batch, heads, seqlen, head_dim)))


def vsa_bwd_workspace_bytes(batch, heads, seqlen, head_dim=HEAD_DIM):
    return int(lib().vsa_bwd_workspace_bytes(make_shape(batch, heads, seqlen, head_dim)))


def vsa_invert_indices(q2k_idx, q2k_num, num_kv_blocks, k2q_idx=None, k2q_num=None, dev_err=None,
                       stream=None):
    """q2k [B,H,nb,topk] / [B,H,nb] int32 -> (k2q_idx [B,H,nb,nb], k2q_num [B,H,nb])."""
    _need(q2k_idx, "q2k_idx", torch.int32, 4)
    _need(q2k_num, "q2k_num", torch.int32, 3)
    B, H, nq, topk = q2k_idx.shape
    nb = int(num_kv_blocks)
    if nq != nb or tuple(q2k_num.shape) != (B, H, nq):
        raise ValueError("q2k_idx/q2k_num shapes do not match num_kv_blocks")
    dev = q2k_idx.device
    if k2q_idx is None:
        k2q_idx = torch.empty((B, H, nb, nb), dtype=torch.int32, device=dev)
    if k2q_num is None:
        k2q_num = torch.empty((B, H, nb), dtype=torch.int32, device=dev)
    _need(k2q_idx, "k2q_idx", torch.int32, 4)
    _need(k2q_num, "k2q_num", torch.int32, 3)
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32)
    _check(lib().vsa_invert_indices(_ptr(q2k_idx), _ptr(q2k_num), topk,
                                    make_shape(B, H, nb * BLOCK), _ptr(k2q_idx), _ptr(k2q_num),
                                    _ptr(dev_err), _stream(stream)), "vsa_invert_indices")
    return k2q_idx, k2q_num


def _activation_shape(q):
    _need(q, "q", torch.bfloat16, 4)
    B, H, S, D = q.shape
    return B, H, S, D


def vsa_fwd(q, k, v, q2k_idx, q2k_num, vbs, sm_scale, o=None, lse=None, workspace=None,
            stream=None):
    """Block-sparse forward.  Returns (o bf16 [B,H,S,128], lse fp32 [B,H,S] in M form)."""
    B, H, S, D = _activation_shape(q)
    for name, t in (("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 4)
        if t.shape != q.shape:
            raise ValueError("%s must have q's shape" % name)
    _need(q2k_idx, "q2k_idx", torch.int32, 4)
    _need(q2k_num, "q2k_num", torch.int32, 3)
    _need(vbs, "vbs", torch.int32, 1)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    shape = make_shape(B, H, S, D, _block_size(S, vbs))
    need = int(lib().vsa_fwd_workspace_bytes(shape))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(lib().vsa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(q2k_idx), _ptr(q2k_num),
                         q2k_idx.shape[-1], _ptr(vbs), float(sm_scale), shape, _ptr(o), _ptr(lse),
                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                         _stream(stream)), "vsa_fwd")
    return o, lse


def _event_handle(ev):
    if ev is None:
        return None
    if ev.cuda_event == 0:      # torch creates the CUDA event lazily, on first record
        ev.record()
    return ctypes.c_void_p(ev.cuda_event)


def vsa_bwd(dout, q, k, v, o, lse, k2q_idx, k2q_num, vbs, sm_scale, dq=None, dk=None, dv=None,
            workspace=None, stream=None, events=None):
    """Block-sparse backward.  Returns (dq, dk, dv) bf16 [B,H,S,128].  ``events``: optional
    dict of torch.cuda.Event (enable_timing) under keys start / before_main / after_main / end,
    recorded around the backward's stages (vsa_bwd_timed)."""
    B, H, S, D = _activation_shape(q)
    for name, t in (("dout", dout), ("k", k), ("v", v), ("o", o)):
        _need(t, name, torch.bfloat16, 4)
        if t.shape != q.shape:
            raise ValueError("%s must have q's shape" % name)
    _need(lse, "lse", torch.float32, 3)
    _need(k2q_num, "k2q_num", torch.int32, 3)
    _need(vbs, "vbs", torch.int32, 1)
    _need(k2q_idx, "k2q_idx", torch.int32)
    max_q = k2q_idx.shape[-1]
    blk = _block_size(S, vbs)
    if k2q_idx.numel() != B * H * (S // blk) * max_q:
        raise ValueError("k2q_idx must hold [B, H, nb, max_q_blocks] entries")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    shape = make_shape(B, H, S, D, blk)
    need = int(lib().vsa_bwd_workspace_bytes(shape))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    args = (_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(k2q_idx),
            _ptr(k2q_num), max_q, _ptr(vbs), float(sm_scale), shape, _ptr(dq), _ptr(dk), _ptr(dv),
            _ptr(workspace), workspace.numel() * workspace.element_size())
    if events is None:
        _check(lib().vsa_bwd(*args, _stream(stream)), "vsa_bwd")
    else:
        ev = VsaBwdEvents(*(_event_handle(events.get(n)) for n in
                            ("start", "before_main", "after_main", "end")))
        _check(lib().vsa_bwd_timed(*args, ctypes.byref(ev), _stream(stream)), "vsa_bwd_timed")
    return dq, dk, dv


def vsa_bwd_no_alloc(dout, q, k, v, o, lse, k2q_idx, k2q_num, vbs, sm_scale, dq=None, dk=None,
                     dv=None, stream=None):
    """vsa_bwd without a workspace argument: the library uses its static scratch array (for
    callers that cannot allocate device memory; see include/vsa.h).  Returns (dq, dk, dv)."""
    B, H, S, D = _activation_shape(q)
    for name, t in (("dout", dout), ("k", k), ("v", v), ("o", o)):
        _need(t, name, torch.bfloat16, 4)
        if t.shape != q.shape:
            raise ValueError("%s must have q's shape" % name)
    _need(lse, "lse", torch.float32, 3)
    _need(k2q_num, "k2q_num", torch.int32, 3)
    _need(vbs, "vbs", torch.int32, 1)
    _need(k2q_idx, "k2q_idx", torch.int32)
    max_q = k2q_idx.shape[-1]
    blk = _block_size(S, vbs)
    if k2q_idx.numel() != B * H * (S // blk) * max_q:
        raise ValueError("k2q_idx must hold [B, H, nb, max_q_blocks] entries")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib().vsa_bwd_no_alloc(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                  _ptr(k2q_idx), _ptr(k2q_num), max_q, _ptr(vbs), float(sm_scale),
                                  make_shape(B, H, S, D, blk), _ptr(dq), _ptr(dk), _ptr(dv),
                                  _stream(stream)), "vsa_bwd_no_alloc")
    return dq, dk, dv


def vsa_set_wait_limit_ns(limit_ns):
    """Time limit of every pipeline wait in kernels launched from now on (0: the default, 4 s).
    Returns the previous limit."""
    return int(lib().vsa_set_wait_limit_ns(int(limit_ns)))


def vsa_work_order(k2q_num, max_q_blocks, block=BLOCK, order=None, stream=None):
    """The backward's work-item order (items sorted by descending clamped k2q count, stable, per
    (b, h) segment): int32 [B * H * nb] of flat item ids."""
    _need(k2q_num, "k2q_num", torch.int32, 3)
    B, H, nb = k2q_num.shape
    if order is None:
        order = torch.empty(B * H * nb, dtype=torch.int32, device=k2q_num.device)
    _need(order, "order", torch.int32, 1)
    if order.numel() != B * H * nb:
        raise ValueError("order must hold B * H * nb entries")
    _check(lib().vsa_work_order(_ptr(k2q_num), int(max_q_blocks),
                                make_shape(B, H, nb * block, HEAD_DIM, block), _ptr(order),
                                _stream(stream)), "vsa_work_order")
    return order


def vsa_bwd_no_alloc_device_error(stream=None):
    """Synchronise the stream and return the device error bits of the last vsa_bwd_no_alloc call
    on the current device."""
    bits = ctypes.c_uint32(0)
    _check(lib().vsa_bwd_no_alloc_device_error(ctypes.byref(bits), _stream(stream)),
           "vsa_bwd_no_alloc_device_error")
    return int(bits.value)


def vsa_read_device_error(workspace, stream=None):
    """Synchronise the stream and return the device error bits of a fwd/bwd workspace."""
    bits = ctypes.c_uint32(0)
    _check(lib().vsa_read_device_error(_ptr(workspace), ctypes.byref(bits), _stream(stream)),
           "vsa_read_device_error")
    return int(bits.value)
