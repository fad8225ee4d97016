"""Float64 CPU oracle (test infrastructure only; see ce_oracle's header)."""

from .ce_oracle import (  # noqa: F401
    LOG2E,
    ce_forward,
    ce_fwd_bwd,
    ce_grad,
    decode_bf16,
    grad_scale,
    linear_ce,
    logsumexp_rows,
    merge_pairs,
    online_lse_sequential,
    round_to_format,
    softmax_rows,
    to_f64,
    ulp,
)
