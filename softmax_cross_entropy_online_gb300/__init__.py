"""GB300-native softmax cross-entropy: online log-sum-exp forward and the fused
in-place backward, as hand-written sm_103a CUDA kernels behind a C ABI.

    from softmax_cross_entropy_online_gb300 import ce_fwd_bwd_inplace
    loss, row_loss, lse = ce_fwd_bwd_inplace(logits, targets)   # logits -> grad

The binding (``api``) needs torch and the in-tree library built by
``build.build()``; ``synthetic`` (seeded inputs) needs only numpy.
"""

__all__ = [
    "ce_forward", "ce_fwd_bwd_inplace", "ce_fwd_bwd_inplace_noalloc", "ce_backward_from_lse",
    "ce_check_errors",
    "ce_max_vocab", "ce_launch_count", "ce_selftest_wait_timeout", "CEError",
    "linear_ce_fwd_bwd", "linear_ce_workspace_size", "ce_gemm_bf16_tn", "ce_gemm_bf16",
    "ce_softmax_forward", "ce_attention_forward",
]


def __getattr__(name):
    if name in __all__:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
