"""Pins of the float64 attention oracle (CPU): closed forms, a library
cross-check, the page's blockwise recurrence against the definition, and a
planted mistake the checks must catch."""

import numpy as np
import pytest

from oracle import attention_oracle as A


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_single_key_gives_its_value():
    # one key: softmax of a single score is 1, so O = V and lse = the score
    q, k, v = rand((2, 3, 1, 8), 1), rand((2, 3, 1, 8), 2), rand((2, 3, 1, 8), 3)
    r = A.attention_forward(q, k, v)
    np.testing.assert_allclose(r["out"], v, rtol=0, atol=1e-15)
    s = np.sum(q * k, axis=-1) / np.sqrt(8)
    np.testing.assert_allclose(r["lse"], s, rtol=0, atol=1e-14)


def test_constant_scores_give_the_mean_of_the_visible_values():
    # zero queries: every score is 0, so each row averages the values it sees:
    # all T values without a mask, values 0..i under the causal mask
    T, D = 13, 16
    q = np.zeros((1, 1, T, D))
    k, v = rand((1, 1, T, D), 4), rand((1, 1, T, D), 5)
    r = A.attention_forward(q, k, v)
    np.testing.assert_allclose(r["out"][0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (T, D)),
                               atol=1e-14)
    np.testing.assert_allclose(r["lse"], np.log(T), atol=1e-14)
    rc = A.attention_forward(q, k, v, A.causal_mask(T))
    running = np.cumsum(v[0, 0], axis=0) / np.arange(1, T + 1)[:, None]
    np.testing.assert_allclose(rc["out"][0, 0], running, atol=1e-14)
    np.testing.assert_allclose(rc["lse"][0, 0], np.log(np.arange(1, T + 1)), atol=1e-14)


def test_causal_mask_matches_the_harness():
    m = A.causal_mask(4)
    assert np.all(m[np.tril_indices(4)] == 0.0)
    assert np.all(np.isneginf(m[np.triu_indices(4, k=1)]))


def test_against_torch_float64_sdpa():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    B, H, T, D = 2, 3, 37, 32
    q, k, v = rand((B, H, T, D), 6), rand((B, H, T, D), 7), rand((B, H, T, D), 8)
    for mask in (None, A.causal_mask(T)):
        r = A.attention_forward(q, k, v, mask)
        tm = None if mask is None else torch.from_numpy(mask)
        ref = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                             torch.from_numpy(v), attn_mask=tm).numpy()
        np.testing.assert_allclose(r["out"], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("block", [1, 7, 16, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_blockwise_recurrence_reaches_the_definition(block, causal):
    B, H, T, D = 1, 2, 45, 16
    q, k, v = rand((B, H, T, D), 9) * 3, rand((B, H, T, D), 10) * 3, rand((B, H, T, D), 11)
    mask = A.causal_mask(T) if causal else None
    d = A.attention_forward(q, k, v, mask)
    b = A.attention_blockwise(q, k, v, mask, block=block)
    np.testing.assert_allclose(b["out"], d["out"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b["lse"], d["lse"], rtol=1e-12, atol=1e-12)


def test_large_score_offsets_stay_finite():
    # scores near 1e4: the running max keeps every exp finite
    T, D = 20, 8
    q = np.full((1, 1, T, D), 100.0)
    k = np.concatenate([np.full((1, 1, T // 2, D), 100.0), np.full((1, 1, T // 2, D), 99.0)],
                       axis=2)
    v = rand((1, 1, T, D), 12)
    d = A.attention_forward(q, k, v)
    b = A.attention_blockwise(q, k, v, block=4)
    assert np.all(np.isfinite(d["out"])) and np.all(np.isfinite(d["lse"]))
    np.testing.assert_allclose(b["out"], d["out"], rtol=1e-12, atol=1e-12)


def test_planted_mistake_dropped_rescale_is_caught(monkeypatch):
    # a recurrence that forgets to rescale the accumulator when the max grows
    # must disagree with the definition on rows whose max rises across blocks
    B, H, T, D = 1, 1, 24, 8
    q, k, v = rand((B, H, T, D), 13) * 4, rand((B, H, T, D), 14) * 4, rand((B, H, T, D), 15)
    real_exp = np.exp

    def broken_blockwise(*args, **kw):
        calls = {"n": 0}

        def exp_without_correction(x):
            calls["n"] += 1
            # the correction factor is the first exp of every block
            return np.ones_like(x) if calls["n"] % 2 == 1 else real_exp(x)

        monkeypatch.setattr(A.np, "exp", exp_without_correction)
        try:
            return A.attention_blockwise(*args, **kw)
        finally:
            monkeypatch.setattr(A.np, "exp", real_exp)

    good = A.attention_forward(q, k, v)
    bad = broken_blockwise(q, k, v, block=4)
    assert not np.allclose(bad["out"], good["out"], rtol=1e-6, atol=1e-6)
