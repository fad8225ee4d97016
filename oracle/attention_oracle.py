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

``attention_blockwise`` is the blockwise form of the same definition, kept
only so that tests can show it reaches the definition's values: every block
of keys gets its own (max, normaliser, accumulator) triple, and the triples
are combined by the associative pairwise merge of the online softmax (the
"This is associative" passage of the "POPCORNBENCH level-1 problem 95
transcript", extended to the value accumulator, which is rescaled by the same
factor as the normaliser).  The flash-attention forward of the Triton
discussion applies that merge one key block after another.

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


def block_triple(s: np.ndarray, v: np.ndarray):
    """(max, normaliser, accumulator) of one block of scores s [..., T, nb] and
    values v [..., nb, D]: m = max_j s_ij, l = sum_j exp(s_ij - m),
    a = sum_j exp(s_ij - m) v_j (a row with no finite score gives (-inf, 0, 0))."""
    m = np.max(s, axis=-1)
    ref = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - ref[..., None])
    return m, np.sum(e, axis=-1), np.einsum("...ij,...jd->...id", e, v)


def merge_triples(x, y):
    """Combine two partial triples: the larger max is kept and each side's
    normaliser and accumulator are rescaled by exp(its max - the larger max)."""
    (m1, l1, a1), (m2, l2, a2) = x, y
    m = np.maximum(m1, m2)
    ref = np.where(np.isfinite(m), m, 0.0)
    f1 = np.exp(m1 - ref)  # exp(-inf) = 0 for a side with no finite score
    f2 = np.exp(m2 - ref)
    return m, f1 * l1 + f2 * l2, f1[..., None] * a1 + f2[..., None] * a2


def attention_blockwise(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask=None,
                        sm_scale: float | None = None, block: int = 16) -> dict:
    """The definition evaluated block by block (test aid): one triple per block
    of `block` keys, merged pairwise (a balanced tree) by merge_triples; the
    output is the merged accumulator over the merged normaliser and lse the
    merged max plus the normaliser's log."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    D = q.shape[-1]
    Tk = k.shape[-2]
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    parts = []
    for j0 in range(0, Tk, block):
        s = np.einsum("...id,...jd->...ij", q, k[..., j0:j0 + block, :]) * sm_scale
        if mask is not None:
            s = s + np.asarray(mask, dtype=np.float64)[:, j0:j0 + block]
        parts.append(block_triple(s, v[..., j0:j0 + block, :]))
    while len(parts) > 1:
        parts = [merge_triples(parts[i], parts[i + 1]) if i + 1 < len(parts) else parts[i]
                 for i in range(0, len(parts), 2)]
    m, l, a = parts[0]
    with np.errstate(invalid="ignore", divide="ignore"):
        out = a / l[..., None]
        lse = np.where(np.isfinite(m), m, 0.0) + np.log(l)
    return {"out": out, "lse": lse}
