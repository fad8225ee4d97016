"""Pins for the float64 oracle: nothing here compares the oracle with itself.

Each test fixes the oracle against something independent of its code: values
printed on the pages, closed forms, invariants the mathematics forces, brute
force on tiny inputs, or a library routine computing the same definition.
The mutation tests at the end plant typical mistakes in copies of the oracle
and check that the pins above catch each of them.
"""

import math
import os

import numpy as np
import pytest

import oracle
from oracle import ce_oracle
from softmax_cross_entropy_online_gb300 import synthetic
from tests.conftest import read_golden

RNG = np.random.default_rng(12345)


# --------------------------------------------------------------------------
# Page-printed values
# --------------------------------------------------------------------------
def test_worked_example_from_transcript(golden_dir):
    g = read_golden(os.path.join(golden_dir, "worked_example_popcornbench_p95.txt"))
    tol = g["printed_tolerance"]
    x = np.array([g["logits"]])
    t = np.array([int(g["target"])])
    f = oracle.ce_forward(x, t, "mean")
    assert abs(f["lse"][0] - g["lse"]) <= tol
    assert abs(f["row_loss"][0] - g["loss"]) <= tol
    assert abs(f["loss"] - g["loss"]) <= tol
    assert abs(math.log(math.exp(f["lse"][0] - 3.0)) - g["log_sum"]) <= tol
    # the page's lane-by-lane merge order: lane0 with lane1, then with lane2
    p = oracle.merge_pairs((1.0, 1.0), (2.0, 1.0))
    assert p[0] == g["merge1_max"] and abs(p[1] - g["merge1_sum"]) <= tol
    p = oracle.merge_pairs(p, (3.0, 1.0))
    assert p[0] == g["merge2_max"] and abs(p[1] - g["merge2_sum"]) <= tol
    # the sequential recurrence reaches the same pair
    m, s = oracle.online_lse_sequential(g["logits"])
    assert m == g["merge2_max"] and abs(s - g["merge2_sum"]) <= tol


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1, 2, 3, 7, 1024, 50257])
@pytest.mark.parametrize("c", [0.0, -7.5, 1e4, -1e4, 88.5])
def test_uniform_logits_give_log_v(V, c):
    # transcript, passage "If all logits are the same value L": loss = log V
    M = 3
    x = np.full((M, V), c)
    t = np.arange(M) % V
    f = oracle.ce_fwd_bwd(x, t, "mean")
    np.testing.assert_allclose(f["row_loss"], math.log(V), rtol=0, atol=1e-12 * max(1, abs(c)))
    expect = np.full((M, V), 1.0 / V)
    expect[np.arange(M), t] -= 1.0
    np.testing.assert_allclose(f["grad"], expect / M, rtol=0, atol=4e-16 * max(1, abs(c)))


@pytest.mark.parametrize("V", [2, 9, 4096, 131072])
def test_one_hot_dominant_row(V):
    x = np.zeros((2, V))
    t = np.array([0, V - 1])
    x[0, 0] = 50.0
    x[1, V - 1] = 50.0
    f = oracle.ce_fwd_bwd(x, t, "sum")
    expect = math.log1p((V - 1) * math.exp(-50.0))
    # exact value ~(V-1)e^-50 is below float64 resolution next to 1: absolute check
    np.testing.assert_allclose(f["row_loss"], expect, rtol=0, atol=1e-15)
    assert f["row_loss"].max() < 1e-15 and f["row_loss"].min() >= 0.0
    # gradient: target entry = p_t - 1 = -(V-1)e^-50 / (1 + (V-1)e^-50)
    q = (V - 1) * math.exp(-50.0)
    np.testing.assert_allclose(f["grad"][0, 0], -q / (1 + q), rtol=0, atol=1e-15)
    np.testing.assert_allclose(f["grad"][0, 1], math.exp(-50.0) / (1 + q), rtol=1e-9)


def test_two_classes_is_softplus():
    d = RNG.normal(0, 5, size=64)
    x = np.stack([np.zeros(64), d], axis=1)
    t = np.zeros(64, dtype=np.int64)
    f = oracle.ce_forward(x, t, "none")
    # lse - x_t cancels for small losses: absolute error ~ eps * |lse|
    err = np.abs(f["row_loss"] - np.logaddexp(0.0, d))
    assert np.all(err <= 1e-13 * np.logaddexp(0.0, d) + 4e-16 * (1 + np.abs(d)))
    assert f["loss"] is None


def test_reductions_and_empty():
    x = RNG.normal(size=(5, 11))
    t = RNG.integers(0, 11, 5)
    fm = oracle.ce_forward(x, t, "mean")
    fs = oracle.ce_forward(x, t, "sum")
    assert abs(fm["loss"] * 5 - fs["loss"]) < 1e-12
    assert abs(fs["loss"] - float(np.sum(fs["row_loss"]))) == 0.0
    e = oracle.ce_forward(np.zeros((0, 7)), np.zeros(0, np.int64), "mean")
    assert math.isnan(e["loss"])
    assert oracle.ce_forward(np.zeros((0, 7)), np.zeros(0, np.int64), "sum")["loss"] == 0.0
    assert oracle.grad_scale("mean", 4) == 0.25 and oracle.grad_scale("sum", 4) == 1.0


def test_out_of_range_target_row():
    x = RNG.normal(size=(4, 6))
    t = np.array([0, 6, -1, 5])
    f = oracle.ce_fwd_bwd(x, t, "sum")
    assert np.isnan(f["row_loss"][1]) and np.isnan(f["row_loss"][2])
    assert np.all(np.isfinite(f["row_loss"][[0, 3]]))
    assert list(f["bad"]) == [False, True, True, False]
    sm = np.exp(x - f["lse"][:, None])
    np.testing.assert_allclose(f["grad"][1], sm[1], rtol=1e-15)
    assert math.isnan(oracle.ce_forward(x, t, "mean")["loss"])


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------
def test_shift_invariance():
    x = RNG.normal(size=(16, 37))
    t = RNG.integers(0, 37, 16)
    c = RNG.uniform(-500, 500, size=(16, 1))
    a = oracle.ce_fwd_bwd(x, t, "mean")
    b = oracle.ce_fwd_bwd(x + c, t, "mean")
    np.testing.assert_allclose(a["row_loss"], b["row_loss"], rtol=0, atol=1e-10)
    np.testing.assert_allclose(a["grad"], b["grad"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(b["lse"], a["lse"] + c[:, 0], rtol=1e-14)


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_gradient_invariants(reduction):
    M, V = 32, 513
    x = RNG.normal(0, 3, size=(M, V))
    t = RNG.integers(0, V, M)
    f = oracle.ce_fwd_bwd(x, t, reduction)
    scale = 1.0 / M if reduction == "mean" else 1.0
    g = f["grad"]
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=V * 1e-16 * scale * 8)
    assert np.all(g <= scale) and np.all(g >= -scale)
    assert np.all(g[np.arange(M), t] < 0)  # only the target entry is negative
    mask = np.ones_like(g, dtype=bool)
    mask[np.arange(M), t] = False
    assert np.all(g[mask] > 0)
    np.testing.assert_allclose(oracle.softmax_rows(x).sum(axis=1), 1.0, rtol=1e-14)
    # row_loss is -log p_target, so it is positive and equals -log(1 + g_t/scale)
    np.testing.assert_allclose(f["row_loss"], -np.log(g[np.arange(M), t] / scale + 1.0),
                               rtol=1e-9)


@pytest.mark.parametrize("M,V", [(1, 2), (2, 3), (3, 5), (4, 9)])
def test_finite_differences(M, V):
    x = RNG.normal(0, 2, size=(M, V))
    t = RNG.integers(0, V, M)
    g = oracle.ce_fwd_bwd(x, t, "mean")["grad"]

    def L(z):
        return oracle.ce_forward(z, t, "mean")["loss"]

    h = 1e-5
    num = np.zeros_like(x)
    for i in range(M):
        for j in range(V):
            xp = x.copy()
            xm = x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            num[i, j] = (L(xp) - L(xm)) / (2 * h)
    np.testing.assert_allclose(g, num, rtol=0, atol=1e-9)


def test_brute_force_tiny():
    # no max subtraction: log(sum exp(x)) - x_t with plain Python loops, |x| <= 20
    M, V = 6, 10
    x = RNG.uniform(-20, 20, size=(M, V))
    t = RNG.integers(0, V, M)
    f = oracle.ce_fwd_bwd(x, t, "mean")
    for i in range(M):
        s = 0.0
        for j in range(V):
            s += math.exp(x[i, j])
        lse = math.log(s)
        assert abs(f["lse"][i] - lse) <= 1e-12 * abs(lse)
        assert abs(f["row_loss"][i] - (lse - x[i, t[i]])) <= 1e-11
        for j in range(V):
            gij = (math.exp(x[i, j]) / s - (1.0 if j == t[i] else 0.0)) / M
            assert abs(f["grad"][i, j] - gij) <= 1e-15


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_library_cross_check_torch_float64(reduction):
    torch = pytest.importorskip("torch")
    M, V = 40, 333
    x = RNG.normal(0, 4, size=(M, V))
    t = RNG.integers(0, V, M)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    ref = torch.nn.functional.cross_entropy(xt, torch.tensor(t), reduction=reduction)
    f = oracle.ce_fwd_bwd(x, t, reduction)
    if reduction == "none":
        np.testing.assert_allclose(f["row_loss"], ref.detach().numpy(), rtol=1e-13)
        ref.sum().backward()
    else:
        assert abs(f["loss"] - ref.item()) <= 1e-13 * abs(ref.item())
        ref.backward()
    scale = 1.0 / M if reduction == "mean" else 1.0
    np.testing.assert_allclose(f["grad"], xt.grad.numpy(), rtol=0, atol=4e-15 * scale)


def test_linear_ce_against_torch_float64():
    torch = pytest.importorskip("torch")
    M, H, V = 12, 16, 50
    h = RNG.normal(size=(M, H))
    W = RNG.normal(0, 0.3, size=(V, H))
    t = RNG.integers(0, V, M)
    f = oracle.linear_ce(h, W, t, "mean")
    ht = torch.tensor(h, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(ht @ Wt.T, torch.tensor(t))
    loss.backward()
    assert abs(f["loss"] - loss.item()) < 1e-13
    np.testing.assert_allclose(f["dH"], ht.grad.numpy(), rtol=0, atol=1e-15)
    np.testing.assert_allclose(f["dW"], Wt.grad.numpy(), rtol=0, atol=1e-15)


def test_linear_ce_equal_weight_rows_closed_form():
    # every row of W equal: each row of logits is constant, so the loss is ln V
    # exactly, G = (1/V - onehot) / M, dH = G W = 0 (G's rows sum to 0) and
    # dW_j = (sum_i h_i / V - sum_{i: t_i = j} h_i) / M
    M, H, V = 6, 5, 7
    rng = np.random.default_rng(7)
    h = rng.normal(size=(M, H))
    W = np.tile(rng.normal(size=H), (V, 1))
    t = np.array([0, 3, 3, 6, 1, 0])
    f = oracle.linear_ce(h, W, t, "mean")
    assert abs(f["loss"] - math.log(V)) < 1e-14
    np.testing.assert_allclose(f["dH"], 0.0, rtol=0, atol=1e-15)
    expect = np.empty((V, H))
    for j in range(V):
        expect[j] = (h.sum(axis=0) / V - h[t == j].sum(axis=0)) / M
    np.testing.assert_allclose(f["dW"], expect, rtol=0, atol=1e-15)


def _linear_ce_fd_ok(fn, M=3, H=4, V=5, seed=8):
    """Central differences of the mean loss against fn's dH and dW."""
    rng = np.random.default_rng(seed)
    h = rng.normal(size=(M, H))
    W = rng.normal(0, 0.5, size=(V, H))
    t = rng.integers(0, V, M)
    f = fn(h, W, t, "mean")
    eps = 1e-6
    ok = True
    for A, dA in ((h, f["dH"]), (W, f["dW"])):
        num = np.zeros_like(A)
        for idx in np.ndindex(A.shape):
            save = A[idx]
            A[idx] = save + eps
            up = oracle.linear_ce(h, W, t, "mean")["loss"]
            A[idx] = save - eps
            dn = oracle.linear_ce(h, W, t, "mean")["loss"]
            A[idx] = save
            num[idx] = (up - dn) / (2 * eps)
        ok = ok and dA.shape == num.shape and np.allclose(dA, num, rtol=0, atol=1e-8)
    return ok


def test_linear_ce_finite_differences():
    assert _linear_ce_fd_ok(oracle.linear_ce)


@pytest.mark.parametrize("kind", ["no_mean_scale", "no_one_hot", "dW_from_W"])
def test_linear_ce_planted_mistakes_are_caught(kind, monkeypatch):
    # each mistake is planted in the oracle (on the CPU) and must fail the
    # finite-difference pin above
    real_grad = ce_oracle.ce_grad

    def broken(h, W, t, reduction="mean"):
        with monkeypatch.context() as mp:
            if kind == "no_mean_scale":
                mp.setattr(ce_oracle, "grad_scale", lambda reduction, M: 1.0)
            elif kind == "no_one_hot":
                mp.setattr(ce_oracle, "ce_grad",
                           lambda x, t_, lse, scale: real_grad(x, np.full_like(t_, -1), lse, scale))
            f = ce_oracle.linear_ce(h, W, t, reduction)
        if kind == "dW_from_W":
            # the weight gradient taken against the wrong operand (W's first M
            # rows in place of h)
            f["dW"] = f["grad"].T @ np.asarray(W, dtype=np.float64)[:len(t)]
        return f

    assert not _linear_ce_fd_ok(broken), kind


def test_online_recurrence_reaches_definition():
    # the streaming pass and any merge tree give the defined lse
    for V in [1, 2, 17, 300]:
        row = RNG.normal(0, 10, size=V)
        m, s = oracle.online_lse_sequential(row)
        lse = oracle.logsumexp_rows(row[None, :])[0]
        assert abs(m + math.log(s) - lse) < 1e-12 * max(1, abs(lse))
        pairs = [(float(v), 1.0) for v in row]
        while len(pairs) > 1:
            pairs = [oracle.merge_pairs(pairs[i], pairs[i + 1]) if i + 1 < len(pairs)
                     else pairs[i] for i in range(0, len(pairs), 2)]
        assert abs(pairs[0][0] + math.log(pairs[0][1]) - lse) < 1e-12 * max(1, abs(lse))
    assert oracle.merge_pairs((-math.inf, 0.0), (-math.inf, 0.0)) == (-math.inf, 0.0)


# --------------------------------------------------------------------------
# Statistical sanity on the workload distributions (catches gross mistakes)
# --------------------------------------------------------------------------
def test_expected_loss_on_gaussian_logits():
    # E[lse] ~= log V + sigma^2/2 for iid N(0, sigma^2) logits; E[x_t] = 0
    x, t = synthetic.make_workload("small_f32_256x1024")
    f = oracle.ce_forward(oracle.to_f64(x, "f32"), t, "mean")
    assert abs(np.mean(f["lse"]) - (math.log(1024) + 0.5)) < 0.02
    assert abs(f["loss"] - (math.log(1024) + 0.5)) < 0.35


def test_expected_lse_on_spiked_rows():
    # 1% of entries at +30 dominate: lse ~= 30 + log(0.01 V)
    w = synthetic.WORKLOADS["f16_8192x131072_spiked"]
    x = synthetic.make_logits(4, w.V, w.dtype, w.sigma, w.spike_prob, w.spike_value, seed=3)
    lse = oracle.logsumexp_rows(oracle.to_f64(x, "f16"))
    assert np.all(np.abs(lse - (30 + math.log(0.01 * w.V))) < 0.15)


# --------------------------------------------------------------------------
# Number-format helpers against library conversions
# --------------------------------------------------------------------------
def _probe_values():
    v = np.concatenate([
        RNG.normal(0, 1, 20000), RNG.normal(0, 1e-6, 5000), RNG.normal(0, 1e-30, 2000),
        RNG.normal(0, 1e4, 2000), np.ldexp(RNG.uniform(1, 2, 3000), RNG.integers(-160, 20, 3000)),
    ])
    # exact ties of each format's spacing near 1 and in the subnormal range
    ties = [1 + 2.0**-11, 1 + 3 * 2.0**-11, 1 + 2.0**-24, 1 + 3 * 2.0**-24, 1 + 2.0**-8,
            1 + 3 * 2.0**-8, 2.0**-25, 3 * 2.0**-25, 2.0**-150, 3 * 2.0**-150, 65520.0, 65519.0]
    return np.concatenate([v, ties, -np.array(ties), [0.0, -0.0]])


@pytest.mark.parametrize("fmt,npt", [("f16", np.float16), ("f32", np.float32)])
def test_round_to_format_matches_numpy(fmt, npt):
    v = _probe_values()
    with np.errstate(over="ignore"):
        ref = v.astype(npt).astype(np.float64)
    got = oracle.round_to_format(v, fmt)
    assert np.array_equal(got, ref, equal_nan=True)


def test_round_to_bf16_matches_bit_encoder():
    # for float32 inputs one RN step either way: compare with the bit-level encoder
    v = _probe_values().astype(np.float32)
    v = v[np.isfinite(v)]
    enc = oracle.decode_bf16(synthetic.f32_to_bf16_bits(v))
    got = oracle.round_to_format(v.astype(np.float64), "bf16")
    assert np.array_equal(got, enc)
    assert oracle.round_to_format(np.array([1 + 2.0**-8]), "bf16")[0] == 1.0  # tie to even
    assert oracle.round_to_format(np.array([1 + 3 * 2.0**-8]), "bf16")[0] == 1 + 2.0**-6


def test_ulp_helper():
    assert oracle.ulp(np.array([1.0]), "f16")[0] == 2.0**-10
    assert oracle.ulp(np.array([0.0]), "f16")[0] == 2.0**-24
    assert oracle.ulp(np.array([2.0**-20]), "f16")[0] == 2.0**-24
    assert oracle.ulp(np.array([1.5]), "bf16")[0] == 2.0**-7
    assert oracle.ulp(np.array([1e-40]), "f32")[0] == 2.0**-149
    assert oracle.ulp(np.array([-3.0]), "f32")[0] == 2.0**-22


# --------------------------------------------------------------------------
# Planted mistakes: each mutated oracle must fail at least one pin above
# --------------------------------------------------------------------------
def _forward_variant(kind):
    def fwd(x, t, reduction="mean"):
        x = np.asarray(x, dtype=np.float64)
        M, V = x.shape
        m = x.max(axis=1)
        if kind == "dropped_max":
            lse = np.log(np.sum(np.exp(x - m[:, None]), axis=1))
        elif kind == "wrong_sign":
            lse = m + np.log(np.sum(np.exp(x - m[:, None]), axis=1))
            lse = -lse
        elif kind == "transposed_index":
            lse = m + np.log(np.sum(np.exp(x - m[:, None]), axis=1))
        elif kind == "log2_not_ln":
            lse = m + np.log2(np.sum(np.exp(x - m[:, None]), axis=1))
        else:
            lse = m + np.log(np.sum(np.exp(x - m[:, None]), axis=1))
        if kind == "transposed_index":
            xt = x[np.arange(M) % V, np.minimum(np.arange(M), V - 1)]
        else:
            xt = x[np.arange(M), t]
        row = lse - xt
        if kind == "mean_over_v":
            loss = float(row.sum() / V)
        else:
            loss = float(row.sum() / M)
        return row, loss

    return fwd


@pytest.mark.parametrize("kind", ["dropped_max", "wrong_sign", "transposed_index",
                                  "log2_not_ln", "mean_over_v"])
def test_planted_mistakes_are_caught(kind, golden_dir):
    fwd = _forward_variant(kind)
    g = read_golden(os.path.join(golden_dir, "worked_example_popcornbench_p95.txt"))
    failures = 0
    # pin 1: page's worked example
    row, loss = fwd(np.array([g["logits"]]), np.array([1]))
    failures += abs(loss - g["loss"]) > g["printed_tolerance"]
    # pin 2: uniform logits with an offset give log V
    x = np.full((3, 5), 4.0)
    row, _ = fwd(x, np.array([0, 1, 2]))
    failures += not np.allclose(row, math.log(5))
    # pin 3: torch float64 cross-entropy on random rows
    torch = pytest.importorskip("torch")
    x = RNG.normal(size=(6, 4))
    t = np.array([3, 0, 1, 2, 3, 1])
    _, loss = fwd(x, t)
    ref = torch.nn.functional.cross_entropy(torch.tensor(x), torch.tensor(t)).item()
    failures += abs(loss - ref) > 1e-12
    assert failures >= 1, f"planted mistake {kind!r} escaped every pin"
    # and the unmutated variant passes them all
    row, loss = _forward_variant("none")(np.array([g["logits"]]), np.array([1]))
    assert abs(loss - g["loss"]) <= g["printed_tolerance"]


def test_softmax_matches_torch_float64():
    torch = pytest.importorskip("torch")
    x = RNG.normal(0, 5, size=(17, 301))
    ref = torch.softmax(torch.tensor(x, dtype=torch.float64), dim=1).numpy()
    np.testing.assert_allclose(oracle.softmax_rows(x), ref, rtol=1e-13, atol=1e-300)


def test_softmax_closed_forms():
    # uniform rows give 1/V for any offset; two classes give the logistic
    # function of the difference; a row with one entry 50 above the rest puts
    # 1 / (1 + (V - 1) e^-50) on it; and rows are shift-invariant
    for V, c in ((1, 0.0), (7, -3.5), (4096, 1e4)):
        # the exponent x - lse carries lse's rounding, up to an ulp of |c| + ln V
        tol = 4 * np.finfo(np.float64).eps * (abs(c) + math.log(V) + 1)
        np.testing.assert_allclose(oracle.softmax_rows(np.full((3, V), c)), 1.0 / V, rtol=tol)
    a = RNG.normal(size=(9, 2)) * 4
    p = oracle.softmax_rows(a)
    np.testing.assert_allclose(p[:, 0], 1.0 / (1.0 + np.exp(a[:, 1] - a[:, 0])), rtol=1e-14)
    V = 1000
    x = np.zeros((1, V))
    x[0, 17] = 50.0
    p = oracle.softmax_rows(x)
    np.testing.assert_allclose(p[0, 17], 1.0 / (1.0 + (V - 1) * math.exp(-50.0)), rtol=1e-15)
    np.testing.assert_allclose(p[0, 0], math.exp(-50.0) / (1.0 + (V - 1) * math.exp(-50.0)),
                               rtol=1e-13)
    x = RNG.normal(size=(5, 33))
    np.testing.assert_allclose(oracle.softmax_rows(x + RNG.normal(size=(5, 1)) * 100),
                               oracle.softmax_rows(x), rtol=1e-12)


@pytest.mark.parametrize("kind", ["unstabilised_lse", "lse_over_columns", "lse_missing_log"])
def test_softmax_planted_mistakes_are_caught(kind, monkeypatch):
    # each mistake is planted in the oracle's log-sum-exp (on the CPU) and must
    # fail the closed forms above
    def unstabilised(x):
        with np.errstate(over="ignore"):
            return np.log(np.sum(np.exp(np.asarray(x, dtype=np.float64)), axis=1))

    def over_columns(x):
        x = np.asarray(x, dtype=np.float64)
        m = np.max(x, axis=0)
        r = m + np.log(np.sum(np.exp(x - m[None, :]), axis=0))
        return np.resize(r, x.shape[0])

    def missing_log(x):
        x = np.asarray(x, dtype=np.float64)
        m = np.max(x, axis=1)
        return m + np.sum(np.exp(x - m[:, None]), axis=1)

    fake = {"unstabilised_lse": unstabilised, "lse_over_columns": over_columns,
            "lse_missing_log": missing_log}[kind]
    monkeypatch.setattr(ce_oracle, "logsumexp_rows", fake)
    with pytest.raises(AssertionError), np.errstate(all="ignore"):
        test_softmax_closed_forms()
