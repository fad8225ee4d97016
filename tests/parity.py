"""Helpers for GPU-vs-oracle parity tests (test infrastructure).

Tolerances (from the stated targets; the arithmetic behind them is in the
design notes):
  * fp32 logits: per-row loss and lse |err| <= 1e-4; reduced loss relative
    error <= 1e-5; gradient |M*g_gpu - M*g_ref| <= 1e-5 (i.e. |g err| <=
    1e-5 * scale).
  * fp16/bf16 logits (fp32 accumulation): per-row loss and lse |err| <= 2e-3;
    gradient within one unit in the last place of the output dtype of the
    float64 reference plus the fp32 evaluation error of softmax, scaled:
    |g_gpu - RN(g_ref)| <= ulp(g_ref) + 4e-6 * scale.  This stays far inside
    the stated bound (2e-3 absolute plus one ulp).
  * lse is an fp32 output: its own rounding, bounded by 2^-22 relative (one
    rounding of the sum m + ln S plus the hardware log2's error), is added to
    the row tolerance.

The 4e-6 * scale term is the absolute error of p = exp(x - lse) in fp32: the
row sum near 1 is rounded at 2^-24 per addition over a few tens of additions
(<= ~70 * 2^-24 = 4.2e-6), and exp2/log2 are evaluated to ~2^-22.  It only
matters where the exact gradient is smaller than that error, e.g. the target
entry of a row whose target dominates (p_t -> 1, g_t -> 0).
"""

from __future__ import annotations

import functools

import numpy as np
import torch

import oracle

ROW_TOL = {"f32": 1e-4, "f16": 2e-3, "bf16": 2e-3}
LOSS_REL_TOL_F32 = 1e-5
GRAD_TOL_F32 = 1e-5  # on M*g (scale-normalised)
GRAD_ABS_EPS = 4e-6  # fp32 evaluation error of softmax, times scale
TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_device(x: np.ndarray, dtype: str, device="cuda", offset_elems: int = 0) -> torch.Tensor:
    """Upload storage-dtype logits; with offset_elems > 0 the tensor starts that
    many elements into a larger buffer (a base pointer off the 16-byte grid)."""
    if dtype == "bf16":
        src = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        src = torch.from_numpy(np.ascontiguousarray(x))
    if offset_elems == 0:
        return src.to(device)
    M, V = x.shape
    buf = torch.empty(M * V + offset_elems, dtype=TORCH_DT[dtype], device=device)
    view = buf[offset_elems:].view(M, V)
    view.copy_(src.to(device))
    return view


def to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def widen(x_storage: np.ndarray, dtype: str) -> np.ndarray:
    return oracle.to_f64(x_storage, dtype)


def check_rows(name, got, ref, tol, rows=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if rows is not None:
        got = got[rows]
    both_nan = np.isnan(got) & np.isnan(ref)
    err = np.where(both_nan, 0.0, np.abs(got - ref))
    bad = ~(err <= tol)
    assert not bad.any(), (f"{name}: {bad.sum()} rows beyond tolerance; worst "
                           f"{np.nanmax(err):.3e} at {int(np.argmax(np.where(np.isnan(err), np.inf, err)))}")


def check_lse(name, got, ref, tol, rows=None):
    ref = np.asarray(ref, dtype=np.float64)
    check_rows(name, got, ref, tol + 2.0**-22 * np.abs(ref), rows)


def check_loss(got: float, ref: float, dtype: str, M: int):
    if np.isnan(ref):
        assert np.isnan(got)
        return
    if dtype == "f32":
        assert abs(got - ref) <= LOSS_REL_TOL_F32 * max(abs(ref), 1e-30) + 1e-7, (got, ref)
    else:
        # the mean of per-row errors bounded by the per-row tolerance
        assert abs(got - ref) <= ROW_TOL[dtype] * max(1.0, 1.0 if M else 0.0), (got, ref)


def check_grad(g_storage: np.ndarray, x64: np.ndarray, t: np.ndarray, lse_ref: np.ndarray,
               scale: float, dtype: str):
    """Compare gradient rows (storage dtype) with the float64 reference rows."""
    g_ref = oracle.ce_grad(x64, t, lse_ref, scale)
    g = oracle.to_f64(g_storage, dtype)
    if dtype == "f32":
        err = np.abs(g - g_ref)
        tol = GRAD_TOL_F32 * abs(scale)
        assert np.all(err <= tol), f"grad: worst |err| {err.max():.3e} > {tol:.3e}"
    else:
        r = oracle.round_to_format(g_ref, dtype)
        err = np.abs(g - r)
        u = oracle.ulp(g_ref, dtype)
        bad = err > u + GRAD_ABS_EPS * abs(scale)
        assert not bad.any(), (f"grad: {bad.sum()} elements beyond 1 ulp; e.g. got {g[bad][:4]} "
                               f"ref {g_ref[bad][:4]}")
        assert np.all(np.abs(g - g_ref) <= 2e-3 + u)


def sample_rows(M: int, n: int, seed: int = 7) -> np.ndarray:
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    rows = rng.choice(M, size=n - 2, replace=False)
    return np.unique(np.concatenate([[0, M - 1], rows]))


def oracle_full_loss(x_storage: np.ndarray, t: np.ndarray, dtype: str, reduction: str = "mean",
                     block: int = 1024) -> float:
    """The float64 oracle's reduced loss over every row of a batch, evaluated in
    row blocks so that a multi-GB workload never widens to float64 at once."""
    M = x_storage.shape[0]
    total = 0.0
    for r0 in range(0, M, block):
        f = oracle.ce_forward(widen(x_storage[r0:r0 + block], dtype), t[r0:r0 + block], "sum")
        total += f["loss"]
    if reduction == "sum":
        return total
    return total / M if M else float("nan")


@functools.lru_cache(maxsize=4)
def workload_full_loss(name: str) -> float:
    """oracle_full_loss of a named workload (mean), computed once per process."""
    from softmax_cross_entropy_online_gb300 import synthetic
    w = synthetic.WORKLOADS[name]
    x, t = synthetic.make_workload(w)
    return oracle_full_loss(x, t, w.dtype)
