"""Float64 CPU oracle for row-wise softmax cross-entropy.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
module.  The library's CUDA path never imports, links or calls it, and this
module imports nothing from the library: the two share no code.

What it computes (sources, cited by page title and passage):

* "POPCORNBENCH level-1 problem 95 transcript" (a CUDA cross-entropy kernel
  for [32768, 4096] fp32): the per-row definition "max, subtract, exp, sum,
  log", i.e. ``loss_i = log sum_j exp(x_ij - m_i) + m_i - x_{i,t_i}``, with
  the default mean reduction over rows.
* "Cross Entropy Loss performance issue" (Triton issue #5509), the
  ``loss_kernel`` listing: the row output is ``log(sumexp) + max - x_target``
  in fp32.
* "9 Triton kernels in 9 weeks", week seven (fused cross-entropy): forward
  and backward in one pass, the gradient written over the logits buffer.
  The gradient of the mean loss is ``(softmax - onehot) / M``.

Every quantity is computed in float64 straight from its definition; the
online (streaming) formulation is *not* used for the reference values.  The
streaming recurrence and its pairwise merge are written out separately
(``online_lse_sequential``, ``merge_pairs``) only so that tests can pin them
to the worked trace on the transcript page and show they reach the same
value as the definition.

Readings taken where the pages are silent (each is repeated in the design
notes):

* mean divides by M (every row counts; no ignore-index, weights or label
  smoothing appear on the pages); M == 0 gives NaN for mean, 0 for sum;
* gradient scale: 1/M for mean, 1 for sum and none;
* a target outside [0, V) makes that row's loss NaN and drops the one-hot
  term from its gradient (the row's gradient is softmax * scale); the
  library additionally raises an error flag;
* the gradient is rounded to the logits' dtype with round-to-nearest-even,
  subnormals kept.

Parity status: every function here is pinned by the tests in
``tests/test_oracle.py`` (page worked example, closed forms, invariants,
finite differences, brute force, and an independent library routine).
"""

from __future__ import annotations

import math

import numpy as np

LOG2E = 1.4426950408889634  # log2(e), the exp -> exp2 identity used on the pages

# ----------------------------------------------------------------------------
# Number formats.  (exponent bits are implied by emin; mant = stored bits)
# ----------------------------------------------------------------------------
_FORMATS = {
    # name: (stored mantissa bits, minimum normal exponent, maximum finite value)
    "f32": (23, -126, float(np.finfo(np.float32).max)),
    "f16": (10, -14, 65504.0),
    "bf16": (7, -126, float.fromhex("0x1.fep127")),
}


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values.

    A bfloat16 is the upper half of an IEEE binary32, so widening is exact.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def to_f64(x: np.ndarray, fmt: str) -> np.ndarray:
    """Exact float64 view of logits stored as fmt ('f32', 'f16', or 'bf16' bits)."""
    if fmt == "bf16":
        return decode_bf16(x)
    return np.asarray(x).astype(np.float64)


def round_to_format(v: np.ndarray, fmt: str) -> np.ndarray:
    """Round float64 values to the nearest value of `fmt` (ties to even).

    Written from the definition of a binary floating-point format: inside a
    binade [2^e, 2^(e+1)) the representable values are spaced 2^(e - mant);
    below the smallest normal 2^emin the spacing stays 2^(emin - mant)
    (subnormals).  Scaling by a power of two is exact in float64, so the
    rounding is one ``np.rint`` (round half to even) on the scaled value.
    Values beyond the largest finite value round to +-inf.
    """
    mant, emin, fmax = _FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    finite = np.isfinite(v) & (v != 0)
    a = v[finite]
    _, e = np.frexp(a)  # a = f * 2^e, 0.5 <= |f| < 1  =>  floor(log2|a|) = e - 1
    q = np.maximum(e - 1, emin) - mant  # exponent of the spacing at |a|
    r = np.ldexp(np.rint(np.ldexp(a, -q)), q)
    # round-to-nearest overflow threshold: fmax + half a spacing of the top binade
    top_half_ulp = math.ldexp(1.0, math.frexp(fmax)[1] - 1 - mant - 1)
    r = np.where(np.abs(a) >= fmax + top_half_ulp, np.copysign(np.inf, a), r)
    out[finite] = r
    return out


def ulp(v: np.ndarray, fmt: str) -> np.ndarray:
    """Spacing of `fmt` at |v| (subnormal spacing below the smallest normal)."""
    mant, emin, _ = _FORMATS[fmt]
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.where(a == 0, 1.0, a))
    q = np.where(a == 0, emin, np.maximum(e - 1, emin)) - mant
    return np.ldexp(np.ones_like(a), q)


# ----------------------------------------------------------------------------
# The method: cross-entropy forward and gradient from the definition.
# ----------------------------------------------------------------------------
def logsumexp_rows(x: np.ndarray) -> np.ndarray:
    """lse_i = m_i + log sum_j exp(x_ij - m_i), with m_i = max_j x_ij.

    The max-subtracted form is the transcript's "per row max, subtract, exp,
    sum, log".  A row whose max is -inf gives NaN (as -inf - (-inf) does);
    that row is outside every tolerance in the tests.
    """
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=1)
    with np.errstate(invalid="ignore", over="ignore"):
        s = np.sum(np.exp(x - m[:, None]), axis=1)
        return m + np.log(s)


def ce_forward(x: np.ndarray, t: np.ndarray, reduction: str = "mean") -> dict:
    """Cross-entropy forward from the definition, in float64.

    Returns ``lse`` [M], ``row_loss`` [M] (= lse_i - x_{i,t_i}; NaN where the
    target is out of range), ``bad`` [M] bool, and ``loss`` (mean: sum/M;
    sum: the sum; none: None).  Sources: the transcript's definition of
    cross-entropy with mean reduction; the loss_kernel output formula of
    "Cross Entropy Loss performance issue".
    """
    x = np.asarray(x, dtype=np.float64)
    t = np.asarray(t, dtype=np.int64)
    M, V = x.shape
    lse = logsumexp_rows(x) if M else np.zeros(0)
    bad = (t < 0) | (t >= V)
    tc = np.where(bad, 0, t)
    xt = x[np.arange(M), tc] if M else np.zeros(0)
    row_loss = np.where(bad, np.nan, lse - xt)
    if reduction == "mean":
        loss = float(np.sum(row_loss) / M) if M else float("nan")
    elif reduction == "sum":
        loss = float(np.sum(row_loss))
    elif reduction == "none":
        loss = None
    else:
        raise ValueError(reduction)
    return {"lse": lse, "row_loss": row_loss, "bad": bad, "loss": loss}


def grad_scale(reduction: str, M: int) -> float:
    """d(loss)/d(row_loss_i): 1/M for mean, 1 for sum and none."""
    if reduction == "mean":
        return 1.0 / M if M else float("nan")
    return 1.0


def ce_grad(x: np.ndarray, t: np.ndarray, lse: np.ndarray, scale: float) -> np.ndarray:
    """g_ij = (exp(x_ij - lse_i) - [j == t_i]) * scale, in float64.

    softmax minus one-hot, times the upstream scale: the gradient the fused
    kernel of "9 Triton kernels in 9 weeks" (week seven) writes over the
    logits.  Rows with an out-of-range target get no one-hot term.
    """
    x = np.asarray(x, dtype=np.float64)
    t = np.asarray(t, dtype=np.int64)
    M, V = x.shape
    with np.errstate(invalid="ignore", over="ignore"):
        p = np.exp(x - np.asarray(lse, dtype=np.float64)[:, None])
    ok = (t >= 0) & (t < V)
    p[np.arange(M)[ok], t[ok]] -= 1.0
    return p * scale


def ce_fwd_bwd(x: np.ndarray, t: np.ndarray, reduction: str = "mean") -> dict:
    """Forward plus the gradient of the reduced loss w.r.t. the logits."""
    f = ce_forward(x, t, reduction)
    M = np.asarray(x).shape[0]
    f["grad"] = ce_grad(x, t, f["lse"], grad_scale(reduction, M))
    return f


def softmax_rows(x: np.ndarray) -> np.ndarray:
    """p_ij = exp(x_ij - lse_i): the fused softmax of "9 Triton kernels in 9
    weeks", week one (three passes fused into one)."""
    x = np.asarray(x, dtype=np.float64)
    lse = logsumexp_rows(x)
    with np.errstate(invalid="ignore", over="ignore"):
        return np.exp(x - lse[:, None])


# ----------------------------------------------------------------------------
# The streaming (online) formulation, written out step by step only so the
# tests can pin it to the transcript's trace.  Not used for reference values.
# ----------------------------------------------------------------------------
def online_lse_sequential(row) -> tuple[float, float]:
    """One pass over a row keeping (running max m, running sum s of exp(x - m)).

    Transcript passage "online softmax algorithm": start from the first
    element with s = 1; a new maximum rescales the old sum by exp(m_old - x)
    and adds 1; otherwise exp(x - m) is added.  Returns (m, s); the row's
    log-sum-exp is m + log s.
    """
    it = iter(float(v) for v in row)
    m = next(it)
    s = 1.0
    for v in it:
        if v > m:
            s = s * math.exp(m - v) + 1.0
            m = v
        else:
            s = s + math.exp(v - m)
    return m, s


def merge_pairs(a: tuple[float, float], b: tuple[float, float]) -> tuple[float, float]:
    """Combine two partial (max, sum) pairs (transcript: "This is associative").

    The sum with the smaller max is rescaled by exp(smaller - larger).
    Two empty partials (-inf, 0) stay empty instead of producing NaN.
    """
    (m1, s1), (m2, s2) = a, b
    if m1 == -math.inf and m2 == -math.inf:
        return (-math.inf, 0.0)
    if m2 > m1:
        return (m2, s2 + s1 * math.exp(m1 - m2))
    return (m1, s1 + s2 * math.exp(m2 - m1))


# ----------------------------------------------------------------------------
# Fused linear + cross-entropy ("9 Triton kernels in 9 weeks", week eight:
# the lm_head projection chunked into the loss so the logits never exist).
# The oracle simply materialises them in float64.
# ----------------------------------------------------------------------------
def linear_ce(h: np.ndarray, W: np.ndarray, t: np.ndarray, reduction: str = "mean") -> dict:
    """logits = h W^T; CE forward; G = dL/dlogits; dH = G W; dW = G^T h (float64)."""
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    logits = h @ W.T
    f = ce_fwd_bwd(logits, t, reduction)
    G = f["grad"]
    f["dH"] = G @ W
    f["dW"] = G.T @ h
    f["logits"] = logits
    return f
