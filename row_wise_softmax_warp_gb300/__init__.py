"""rowops on GB300: row-wise normalise-and-reduce ops (softmax and its backward,
scaled causal attention softmax, hard-masked softmax, logsumexp, fused softmax
cross-entropy, LayerNorm forward/backward, top-k kept mask) as hand-written
sm_103a CUDA kernels behind a C ABI (include/rowops.h).

The functions below are the ctypes binding of that ABI; ``inputs`` holds the
seeded synthetic workloads and ``build`` compiles the library.
"""
from .binding import (  # noqa: F401
    RowopsError,
    library,
    rowops_argmax_onehot,
    rowops_attn_softmax_bwd,
    rowops_attn_softmax_fwd,
    rowops_column_sums,
    rowops_kernel_launches,
    rowops_layernorm_bwd,
    rowops_layernorm_bwd_workspace,
    rowops_layernorm_fwd,
    rowops_logsumexp,
    rowops_lrp_softmax_rows,
    rowops_masked_softmax,
    rowops_masked_softmax_fmask,
    rowops_rmsnorm_bwd,
    rowops_rmsnorm_fwd,
    rowops_router_masked_topk,
    rowops_softmax_bwd,
    rowops_softmax_ce,
    rowops_soft_ce,
    rowops_softmax_fwd,
    rowops_teacher_ce,
    rowops_top_k_rows,
    rowops_topk_kept,
)
