"""Pins of the float64 attention oracle (CPU): closed forms, a library
cross-check, the blockwise (pairwise-merge) form against the definition, and a
planted mistake the checks must catch."""

import numpy as np
import pytest

from oracle import attention_oracle as A


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def pin_single_key(fwd=A.attention_forward):
    # one key: softmax of a single score is 1, so O = V and lse = the score
    q, k, v = rand((2, 3, 1, 8), 1), rand((2, 3, 1, 8), 2), rand((2, 3, 1, 8), 3)
    r = fwd(q, k, v)
    np.testing.assert_allclose(r["out"], v, rtol=0, atol=1e-15)
    s = np.sum(q * k, axis=-1) / np.sqrt(8)
    np.testing.assert_allclose(r["lse"], s, rtol=0, atol=1e-14)


def pin_constant_scores(fwd=A.attention_forward):
    # zero queries: every score is 0, so each row averages the values it sees:
    # all T values without a mask, values 0..i under the causal mask
    T, D = 13, 16
    q = np.zeros((1, 1, T, D))
    k, v = rand((1, 1, T, D), 4), rand((1, 1, T, D), 5)
    r = fwd(q, k, v)
    np.testing.assert_allclose(r["out"][0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (T, D)),
                               atol=1e-14)
    np.testing.assert_allclose(r["lse"], np.log(T), atol=1e-14)
    rc = fwd(q, k, v, A.causal_mask(T))
    running = np.cumsum(v[0, 0], axis=0) / np.arange(1, T + 1)[:, None]
    np.testing.assert_allclose(rc["out"][0, 0], running, atol=1e-14)
    np.testing.assert_allclose(rc["lse"][0, 0], np.log(np.arange(1, T + 1)), atol=1e-14)


def pin_torch_float64_sdpa(fwd=A.attention_forward):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    B, H, T, D = 2, 3, 37, 32
    q, k, v = rand((B, H, T, D), 6), rand((B, H, T, D), 7), rand((B, H, T, D), 8)
    for mask in (None, A.causal_mask(T)):
        r = fwd(q, k, v, mask)
        tm = None if mask is None else torch.from_numpy(mask)
        ref = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                             torch.from_numpy(v), attn_mask=tm).numpy()
        np.testing.assert_allclose(r["out"], ref, rtol=1e-12, atol=1e-12)


def pin_large_score_offsets(fwd=A.attention_forward):
    # scores near 1e4: the max taken out before exp keeps every exp finite, and
    # the result equals the same attention with the offset removed
    T, D = 20, 8
    q = np.full((1, 1, T, D), 100.0)
    k = np.concatenate([np.full((1, 1, T // 2, D), 100.0), np.full((1, 1, T // 2, D), 99.0)],
                       axis=2)
    v = rand((1, 1, T, D), 12)
    r = fwd(q, k, v)
    assert np.all(np.isfinite(r["out"])) and np.all(np.isfinite(r["lse"]))
    # scores are 100 * 100 * 8 / sqrt(8) for the first half of the keys and
    # 99 / 100 of that for the second: weights 1 and exp(-0.01 * that)
    s_hi = 100.0 * 100.0 * D / np.sqrt(D)
    w_lo = np.exp(-0.01 * s_hi)
    expect = (v[0, 0, :T // 2].sum(axis=0) + w_lo * v[0, 0, T // 2:].sum(axis=0)) / (
        T // 2 * (1 + w_lo))
    np.testing.assert_allclose(r["out"][0, 0], np.broadcast_to(expect, (T, D)), rtol=1e-12,
                               atol=1e-12)


PINS = [pin_single_key, pin_constant_scores, pin_torch_float64_sdpa, pin_large_score_offsets]


def test_single_key_gives_its_value():
    pin_single_key()


def test_constant_scores_give_the_mean_of_the_visible_values():
    pin_constant_scores()


def test_causal_mask_matches_the_harness():
    m = A.causal_mask(4)
    assert np.all(m[np.tril_indices(4)] == 0.0)
    assert np.all(np.isneginf(m[np.triu_indices(4, k=1)]))


def test_against_torch_float64_sdpa():
    pin_torch_float64_sdpa()


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
    pin_large_score_offsets()
    T, D = 20, 8
    q = np.full((1, 1, T, D), 100.0)
    k = np.concatenate([np.full((1, 1, T // 2, D), 100.0), np.full((1, 1, T // 2, D), 99.0)],
                       axis=2)
    v = rand((1, 1, T, D), 12)
    d = A.attention_forward(q, k, v)
    b = A.attention_blockwise(q, k, v, block=4)
    np.testing.assert_allclose(b["out"], d["out"], rtol=1e-12, atol=1e-12)


def test_planted_mistake_dropped_rescale_is_caught(monkeypatch):
    # a merge that forgets to rescale the side with the smaller max must disagree
    # with the definition on rows whose max differs between key blocks
    B, H, T, D = 1, 1, 24, 8
    q, k, v = rand((B, H, T, D), 13) * 4, rand((B, H, T, D), 14) * 4, rand((B, H, T, D), 15)

    def merge_without_rescale(x, y):
        (m1, l1, a1), (m2, l2, a2) = x, y
        return np.maximum(m1, m2), l1 + l2, a1 + a2

    good = A.attention_forward(q, k, v)
    monkeypatch.setattr(A, "merge_triples", merge_without_rescale)
    bad = A.attention_blockwise(q, k, v, block=4)
    assert not np.allclose(bad["out"], good["out"], rtol=1e-6, atol=1e-6)
    assert not np.allclose(bad["lse"], good["lse"], rtol=1e-6, atol=1e-6)


def mutated_forward(kind):
    """attention_forward with one plausible mistake planted in it (numpy patched
    only while the oracle runs)."""
    real = {n: getattr(np, n) for n in ("einsum", "sqrt", "max", "asarray", "sum")}

    def fwd(q, k, v, mask=None, sm_scale=None):
        patch = {}
        if kind == "transposed_scores":
            def einsum(spec, *ops, **kw):
                r = real["einsum"](spec, *ops, **kw)
                return r.swapaxes(-1, -2) if spec == "...id,...jd->...ij" else r
            patch["einsum"] = einsum
        elif kind == "inverted_scale":
            patch["sqrt"] = lambda x: 1.0 / real["sqrt"](x)
        elif kind == "negated_mask":
            patch["asarray"] = lambda a, *args, **kw: (
                -real["asarray"](a, *args, **kw) if a is mask else real["asarray"](a, *args, **kw))
        elif kind == "dropped_max":
            patch["max"] = lambda a, *args, **kw: np.zeros_like(real["max"](a, *args, **kw))
        elif kind == "normaliser_over_queries":
            def sum_(a, *args, axis=None, **kw):
                return real["sum"](a, *args, axis=-2 if axis == -1 else axis, **kw)
            patch["sum"] = sum_
        for n, f in patch.items():
            setattr(np, n, f)
        try:
            return A.attention_forward(q, k, v, mask, sm_scale)
        finally:
            for n in patch:
                setattr(np, n, real[n])
    return fwd


@pytest.mark.parametrize("kind", ["transposed_scores", "inverted_scale", "negated_mask",
                                  "dropped_max", "normaliser_over_queries"])
def test_planted_mistakes_in_the_oracle_fail_a_pin(kind):
    pytest.importorskip("torch")
    fwd = mutated_forward(kind)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(fwd)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {kind}"
