"""Float64 CPU oracle for the blockwise attention forward.

TEST INFRASTRUCTURE ONLY (the same rule as ce_oracle: only the tests, the
smoke check and the CPU-baseline leg of the benchmark may import it; the
library never does, and nothing here comes from the library).

What it computes -- "How to optimize an existing Triton Kernel to make it
faster?" (Triton discussion #8261), the flash-attention-2 forward listing and
its test harness: for queries, keys and values of shape [B, NH, T, D], an
additive mask [T, T] (the harness builds a causal one: 0 on and below the
diagonal, -inf above) and ``sm_scale = 1 / sqrt(D)``,

    S = (Q K^T) * sm_scale + mask,   P = softmax_rows(S),   O = P V,

with ``lse = log sum_j exp(S_ij)`` per query row (the value a backward pass
needs; the listing keeps it as the running max plus the log of the running
normaliser).  ``attention_forward`` is this definition, evaluated directly in
float64 (a row of all -inf scores gives NaN, as the definition does).

``attention_blockwise`` restates the listing's algorithm -- blocks of keys,
a running row max, a running normaliser rescaled by ``exp(old max - new
max)``, an output accumulator rescaled by the same factor, one division at the
end -- only so that tests can show it reaches the definition's values.

Parity status: pinned by tests/test_attention_oracle.py (closed forms for one
key and for constant scores, a float64 library cross-check, the blockwise
recurrence against the definition, and a planted mistake).
"""

from __future__ import annotations

import numpy as np


def causal_mask(T: int) -> np.ndarray:
    """The harness's mask: 0 where key j <= query i, -inf above the diagonal."""
    m = np.zeros((T, T), dtype=np.float64)
    m[np.triu_indices(T, k=1)] = -np.inf
    return m


def attention_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask=None,
                      sm_scale: float | None = None) -> dict:
    """O = softmax(Q K^T * sm_scale + mask) V and lse per query row, float64.

    q, k, v: [..., T, D] (any leading batch/head axes); mask: [T, T] or None.
    Returns {"out": [..., T, D], "lse": [..., T]}.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    D = q.shape[-1]
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    s = np.einsum("...id,...jd->...ij", q, k) * sm_scale
    if mask is not None:
        s = s + np.asarray(mask, dtype=np.float64)
    m = np.max(s, axis=-1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        e = np.exp(s - m)
        den = np.sum(e, axis=-1, keepdims=True)
        p = e / den
        out = np.einsum("...ij,...jd->...id", p, v)
        lse = (m + np.log(den))[..., 0]
    return {"out": out, "lse": lse}


def attention_blockwise(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask=None,
                        sm_scale: float | None = None, block: int = 16) -> dict:
    """The listing's blockwise recurrence over key blocks, in float64 (test aid).

    For each block of `block` keys: the block's scores, the new running max,
    the correction exp(old max - new max) applied to the running normaliser
    and to the output accumulator, then the block's exp-scores added to both;
    the output is divided by the normaliser once at the end.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, D = q.shape[-2], q.shape[-1]
    Tk = k.shape[-2]
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    lead = q.shape[:-2]
    run_max = np.full(lead + (T,), -np.inf)
    run_norm = np.zeros(lead + (T,))
    acc = np.zeros(lead + (T, D))
    for j0 in range(0, Tk, block):
        kb = k[..., j0:j0 + block, :]
        vb = v[..., j0:j0 + block, :]
        s = np.einsum("...id,...jd->...ij", q, kb) * sm_scale
        if mask is not None:
            s = s + np.asarray(mask, dtype=np.float64)[:, j0:j0 + block]
        new_max = np.maximum(run_max, np.max(s, axis=-1))
        # -inf - -inf would be NaN: a row with no finite score so far keeps 0
        ref = np.where(np.isfinite(new_max), new_max, 0.0)
        corr = np.exp(np.where(np.isfinite(run_max), run_max - ref, -np.inf))
        e = np.exp(s - ref[..., None])
        run_norm = corr * run_norm + np.sum(e, axis=-1)
        acc = corr[..., None] * acc + np.einsum("...ij,...jd->...id", e, vb)
        run_max = new_max
    with np.errstate(invalid="ignore", divide="ignore"):
        out = acc / run_norm[..., None]
        lse = np.where(np.isfinite(run_max), run_max, 0.0) + np.log(run_norm)
    return {"out": out, "lse": lse}
