"""GB300 (sm_103a) block-sparse video attention: k2q inversion, forward and backward of
64-token block-sparse attention behind a C ABI (include/vsa.h, libvsa.so).

    from block_sparse_video_tok_gb300 import vsa
    k2q_idx, k2q_num = vsa.vsa_invert_indices(q2k_idx, q2k_num, nb)
    o, lse = vsa.vsa_fwd(q, k, v, q2k_idx, q2k_num, vbs, sm_scale)
    dq, dk, dv = vsa.vsa_bwd(do, q, k, v, o, lse, k2q_idx, k2q_num, vbs, sm_scale)

    from block_sparse_video_tok_gb300.autograd import block_sparse_attention
    o = block_sparse_attention(q, k, v, q2k_idx, q2k_num, vbs)   # differentiable in q, k, v
"""
from . import autograd, build, vsa, workloads  # noqa: F401

__all__ = ["autograd", "build", "vsa", "workloads"]
