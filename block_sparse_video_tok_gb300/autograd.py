"""torch.autograd binding of the block-sparse attention path.

`block_sparse_attention(q, k, v, q2k_idx, q2k_num, vbs, sm_scale)` returns O and records, for
the backward, what the backward kernels consume: Q, K, V, O and the base-2 lse (M form) of the
forward.  The backward inverts the selection (q2k -> k2q) and runs the backward kernels, the
order the FastVideo autograd path uses (block_sparse_attn_bwd_sm100a.py,
block_sparse_attn_backward_sm100a: invert_indices, then the sm_100a backward; the custom op's
backward in the compare page main...vsa_bwd_fix, _backward_sm100a).

Argument marshalling only: every step runs in libvsa.so's kernels through `vsa`.
"""
import torch

from . import vsa


class BlockSparseAttention(torch.autograd.Function):
    """O = block-sparse softmax(Q K^T * sm_scale) V over 64-token blocks.

    Inputs: bf16 [B, H, S, 128] q, k, v (S = 64 * nb); int32 q2k_idx [B, H, nb, topk] and q2k_num
    [B, H, nb] (the kv blocks each q block attends to, a set: duplicates count once); int32 vbs
    [nb] (valid tokens of each kv block, <= 64); sm_scale.  Outputs O (bf16, same shape as q)
    and lse (fp32 [B, H, S], not differentiable).  Gradients flow to q, k and v; dq and dk carry
    sm_scale, dv does not.
    """

    @staticmethod
    def forward(ctx, q, k, v, q2k_idx, q2k_num, vbs, sm_scale):
        o, lse = vsa.vsa_fwd(q, k, v, q2k_idx, q2k_num, vbs, sm_scale)
        ctx.save_for_backward(q, k, v, o, lse, q2k_idx, q2k_num, vbs)
        ctx.sm_scale = sm_scale
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse, q2k_idx, q2k_num, vbs = ctx.saved_tensors
        k2q_idx, k2q_num = vsa.vsa_invert_indices(q2k_idx, q2k_num, vbs.numel())
        dq, dk, dv = vsa.vsa_bwd(do.contiguous(), q, k, v, o, lse, k2q_idx, k2q_num, vbs,
                                 ctx.sm_scale)
        return dq, dk, dv, None, None, None, None


def block_sparse_attention(q, k, v, q2k_idx, q2k_num, vbs, sm_scale=None):
    """O of block-sparse attention, differentiable in q, k and v (see BlockSparseAttention).
    sm_scale defaults to 1/sqrt(head_dim)."""
    if sm_scale is None:
        sm_scale = q.shape[-1] ** -0.5
    o, _ = BlockSparseAttention.apply(q, k, v, q2k_idx, q2k_num, vbs, float(sm_scale))
    return o
