"""torch.autograd binding of the block-sparse attention path.

`block_sparse_attention(q, k, v, q2k_idx, q2k_num, vbs, sm_scale)` returns O and records, for
the backward, what the backward kernels consume: Q, K, V, O, the base-2 lse (M form) of the
forward, and the inverted selection k2q.  The FastVideo autograd path inverts the selection
(q2k -> k2q) right before its sm_100a backward (block_sparse_attn_bwd_sm100a.py,
block_sparse_attn_backward_sm100a; the custom op's backward in the compare page
main...vsa_bwd_fix, _backward_sm100a); here the forward does it once and saves the result, so
the backward starts on its preprocess at once, and a caller whose layers share one selection can
invert it once for all of them (`k2q=` below).

Argument marshalling only: every step runs in libvsa.so's kernels through `vsa`.
"""
import torch

from . import vsa


class BlockSparseAttention(torch.autograd.Function):
    """O = block-sparse softmax(Q K^T * sm_scale) V over 64- or 128-token blocks.

    Inputs: bf16 [B, H, S, 128] q, k, v (S = block * nb); int32 q2k_idx [B, H, nb, topk] and
    q2k_num [B, H, nb] (the kv blocks each q block attends to, a set: duplicates count once);
    int32 vbs [nb] (valid tokens of each kv block); sm_scale; k2q_idx / k2q_num: the inverted
    selection (vsa_invert_indices of q2k), or None to invert it here.  Outputs O (bf16, same
    shape as q) and lse (fp32 [B, H, S], not differentiable).  Gradients flow to q, k and v; dq
    and dk carry sm_scale, dv does not.
    """

    @staticmethod
    def forward(ctx, q, k, v, q2k_idx, q2k_num, vbs, sm_scale, k2q_idx=None, k2q_num=None):
        o, lse = vsa.vsa_fwd(q, k, v, q2k_idx, q2k_num, vbs, sm_scale)
        if k2q_idx is None or k2q_num is None:
            k2q_idx, k2q_num = vsa.vsa_invert_indices(q2k_idx, q2k_num, vbs.numel())
        ctx.save_for_backward(q, k, v, o, lse, k2q_idx, k2q_num, vbs)
        ctx.sm_scale = sm_scale
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse, k2q_idx, k2q_num, vbs = ctx.saved_tensors
        dq, dk, dv = vsa.vsa_bwd(do.contiguous(), q, k, v, o, lse, k2q_idx, k2q_num, vbs,
                                 ctx.sm_scale)
        return dq, dk, dv, None, None, None, None, None, None


def block_sparse_attention(q, k, v, q2k_idx, q2k_num, vbs, sm_scale=None, k2q=None):
    """O of block-sparse attention, differentiable in q, k and v (see BlockSparseAttention).
    sm_scale defaults to 1/sqrt(head_dim).  k2q: optional (k2q_idx, k2q_num) of this selection,
    from vsa.vsa_invert_indices, for callers that reuse one selection in several calls; without
    it the forward inverts the selection once and saves it for the backward."""
    if sm_scale is None:
        sm_scale = q.shape[-1] ** -0.5
    k2q_idx, k2q_num = k2q if k2q is not None else (None, None)
    o, _ = BlockSparseAttention.apply(q, k, v, q2k_idx, q2k_num, vbs, float(sm_scale), k2q_idx,
                                      k2q_num)
    return o
