"""The seeded input generator: determinism, dtype encoding, distributions."""

import numpy as np

from softmax_cross_entropy_online_gb300 import synthetic


def test_deterministic_and_blockwise_equal():
    a = synthetic.make_logits(37, 129, "f32", seed=5, block_rows=7)
    b = synthetic.make_logits(37, 129, "f32", seed=5, block_rows=37)
    assert np.array_equal(a, b)
    c = synthetic.make_logits(37, 129, "f32", seed=6)
    assert not np.array_equal(a, c)
    assert np.array_equal(synthetic.make_targets(50, 9, 1), synthetic.make_targets(50, 9, 1))


def test_distributions():
    x = synthetic.make_logits(64, 4096, "f32", sigma=2.0, seed=0).astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 2.0) < 0.02
    s = synthetic.make_logits(64, 4096, "f16", sigma=2.0, spike_prob=0.01, spike_value=30.0)
    frac = np.mean(s == np.float16(30.0))
    assert 0.008 < frac < 0.012
    t = synthetic.make_targets(100000, 50257)
    assert t.min() >= 0 and t.max() < 50257 and t.dtype == np.int64
    assert abs(t.mean() - 50256 / 2) < 500


def test_bf16_encoding_round_to_nearest_even():
    v = np.array([1.0, 1 + 2**-8, 1 + 3 * 2**-8, -2.5, 3.0e38, 1e-40], dtype=np.float32)
    bits = synthetic.f32_to_bf16_bits(v)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1 + 2**-6 and back[3] == -2.5
    assert bits.dtype == np.uint16


def test_workload_table():
    w = synthetic.WORKLOADS["bf16_16384x50257"]
    assert (w.M, w.V, w.dtype, w.sigma) == (16384, 50257, "bf16", 8.0)
    x, t = synthetic.make_workload(w, M=4, V=33)
    assert x.shape == (4, 33) and x.dtype == np.uint16 and t.shape == (4,)
