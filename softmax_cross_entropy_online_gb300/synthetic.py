"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no cross-entropy arithmetic: it only draws logits and
targets with the shapes and value distributions of the workloads the pages
measure, and encodes them in the storage dtype.  Both the CUDA path (which
receives the bytes) and the float64 oracle (which widens the same bytes)
consume its output, so the two sides always see bit-identical inputs.

Generators: numpy's PCG64, one independent substream per quantity (logits,
spike mask, targets) spawned from ``SeedSequence(seed)``.  Drawing in row
blocks consumes the stream in order, so a block-wise draw is identical to a
single draw.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# element sizes of the storage dtypes
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclass(frozen=True)
class Workload:
    """A named synthetic cross-entropy workload."""

    name: str
    M: int
    V: int
    dtype: str  # 'f32' | 'f16' | 'bf16'
    sigma: float  # logits ~ N(0, sigma^2)
    spike_prob: float = 0.0  # per-entry probability of replacing the value
    spike_value: float = 0.0
    seed: int = 0
    desc: str = ""


# The workloads (rows x classes, dtype, distribution).  Targets are uniform
# in [0, V) for all of them.
WORKLOADS = {
    "small_f32_256x1024": Workload(
        "small_f32_256x1024", 256, 1024, "f32", 1.0,
        desc="fp32 [256, 1024], N(0,1); forward only, per-row loss + mean"),
    "f32_32768x4096": Workload(
        "f32_32768x4096", 32768, 4096, "f32", 1.0,
        desc="fp32 [32768, 4096], N(0,1); forward mean, then fwd+bwd in place"),
    "f16_8192x131072_spiked": Workload(
        "f16_8192x131072_spiked", 8192, 131072, "f16", 2.0, 0.01, 30.0,
        desc="fp16 [8192, 131072], N(0, 2^2) with 1% of entries set to +30; fwd+bwd in place"),
    "bf16_16384x50257": Workload(
        "bf16_16384x50257", 16384, 50257, "bf16", 8.0,
        desc="bf16 [16384, 50257] (odd V), N(0,1) x 8; fwd+bwd in place"),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def _streams(seed: int):
    ss = np.random.SeedSequence(seed)
    logit_ss, spike_ss, target_ss = ss.spawn(3)
    return (np.random.Generator(np.random.PCG64(logit_ss)),
            np.random.Generator(np.random.PCG64(spike_ss)),
            np.random.Generator(np.random.PCG64(target_ss)))


def make_logits(M: int, V: int, dtype: str, sigma: float = 1.0,
                spike_prob: float = 0.0, spike_value: float = 0.0,
                seed: int = 0, block_rows: int | None = None) -> np.ndarray:
    """Draw [M, V] logits ~ N(0, sigma^2) (float32 draws scaled by sigma),
    optionally replacing each entry by `spike_value` with probability
    `spike_prob`, then round to the storage dtype (RN-even).

    Returns float32 / float16 arrays, or uint16 bit patterns for bf16.
    """
    g_logit, g_spike, _ = _streams(seed)
    out_dtype = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]
    out = np.empty((M, V), dtype=out_dtype)
    if block_rows is None:
        block_rows = max(1, (1 << 24) // max(V, 1))
    for r0 in range(0, M, block_rows):
        r1 = min(M, r0 + block_rows)
        z = g_logit.standard_normal((r1 - r0, V), dtype=np.float32)
        if sigma != 1.0:
            z *= np.float32(sigma)
        if spike_prob > 0.0:
            mask = g_spike.random((r1 - r0, V), dtype=np.float32) < np.float32(spike_prob)
            z[mask] = np.float32(spike_value)
        if dtype == "f32":
            out[r0:r1] = z
        elif dtype == "f16":
            out[r0:r1] = z.astype(np.float16)
        else:
            out[r0:r1] = f32_to_bf16_bits(z)
    return out


def make_targets(M: int, V: int, seed: int = 0) -> np.ndarray:
    """int64 targets uniform in [0, V)."""
    _, _, g_t = _streams(seed)
    return g_t.integers(0, V, size=M, dtype=np.int64)


def make_workload(w: Workload | str, M: int | None = None, V: int | None = None):
    """(logits, targets) for a named workload, optionally resized."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    M = w.M if M is None else M
    V = w.V if V is None else V
    x = make_logits(M, V, w.dtype, w.sigma, w.spike_prob, w.spike_value, w.seed)
    t = make_targets(M, V, w.seed)
    return x, t


def make_linear_ce_inputs(M: int, H: int, V: int, seed: int = 0):
    """bf16 hidden [M, H] ~ N(0,1), bf16 weight [V, H] ~ N(0, 0.02^2), int64
    targets uniform in [0, V); returned as bf16 bit patterns + int64."""
    ss = np.random.SeedSequence(seed)
    hs, ws, ts = ss.spawn(3)
    gh = np.random.Generator(np.random.PCG64(hs))
    gw = np.random.Generator(np.random.PCG64(ws))
    gt = np.random.Generator(np.random.PCG64(ts))
    h = f32_to_bf16_bits(gh.standard_normal((M, H), dtype=np.float32))
    W = np.empty((V, H), dtype=np.uint16)
    blk = max(1, (1 << 24) // H)
    for r0 in range(0, V, blk):
        r1 = min(V, r0 + blk)
        W[r0:r1] = f32_to_bf16_bits(gw.standard_normal((r1 - r0, H), dtype=np.float32)
                                    * np.float32(0.02))
    t = gt.integers(0, V, size=M, dtype=np.int64)
    return h, W, t


def make_attention_inputs(B: int, NH: int, T: int, D: int, seed: int = 0,
                          q_sigma: float = 1.0):
    """Queries, keys and values [B, NH, T, D] ~ N(0, 1) (queries N(0, q_sigma^2)),
    the distribution of the flash-attention page's harness; bf16 bit patterns."""
    gq, gk, gv = (np.random.Generator(np.random.PCG64(s))
                  for s in np.random.SeedSequence(seed).spawn(3))
    shape = (B, NH, T, D)
    q = gq.standard_normal(shape, dtype=np.float32)
    if q_sigma != 1.0:
        q *= np.float32(q_sigma)
    return (f32_to_bf16_bits(q), f32_to_bf16_bits(gk.standard_normal(shape, dtype=np.float32)),
            f32_to_bf16_bits(gv.standard_normal(shape, dtype=np.float32)))


def make_attention_mask(T: int, seed: int = 0, sigma: float = 1.0,
                        hide_prob: float = 0.0) -> np.ndarray:
    """An additive fp32 mask [T, T] ~ N(0, sigma^2) whose off-diagonal entries
    are -inf with probability `hide_prob` (the diagonal stays finite, so every
    query sees at least one key)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(2)[1]))
    m = g.standard_normal((T, T), dtype=np.float32) * np.float32(sigma)
    if hide_prob > 0.0:
        hide = g.random((T, T), dtype=np.float32) < np.float32(hide_prob)
        np.fill_diagonal(hide, False)
        m[hide] = -np.inf
    return m
