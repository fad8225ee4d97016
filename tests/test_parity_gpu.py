"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle,
element by element, on seeded synthetic inputs."""

import math
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from softmax_cross_entropy_online_gb300 import synthetic  # noqa: E402
from tests import parity as P  # noqa: E402

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(2024)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_online_gb300 import api, build
    build.build()
    api.lib()
    yield


def api():
    from softmax_cross_entropy_online_gb300 import api as a
    return a


def run_all(x_np, t_np, dtype, reduction="mean", offset_elems=0, stream=None):
    """Run the forward and the fused fwd+bwd on the same input."""
    a = api()
    t_dev = torch.from_numpy(t_np).cuda()
    xf = P.to_device(x_np, dtype, offset_elems=offset_elems)
    loss_f, rl_f, lse_f = a.ce_forward(xf, t_dev, reduction, stream=stream)
    xb = P.to_device(x_np, dtype, offset_elems=offset_elems)
    loss_b, rl_b, lse_b = a.ce_fwd_bwd_inplace(xb, t_dev, reduction, stream=stream)
    M = x_np.shape[0]
    scale = oracle.grad_scale(reduction, M) if M else 1.0
    torch.cuda.synchronize()
    return dict(loss_f=loss_f, rl_f=rl_f, lse_f=lse_f, loss_b=loss_b, rl_b=rl_b, lse_b=lse_b,
                grad_b=xb, scale=scale)


def check_backward_from_lse(x_rows, t_rows, lse_ref, scale, dtype, offset_elems=0):
    """ce_backward_from_lse on the given rows, fed the oracle's lse rounded to
    fp32; the reference gradient uses that same fp32 lse."""
    a = api()
    lse32 = lse_ref.astype(np.float32)
    xl = P.to_device(x_rows, dtype, offset_elems=offset_elems)
    a.ce_backward_from_lse(xl, torch.from_numpy(t_rows).cuda(), torch.from_numpy(lse32).cuda(),
                           scale)
    torch.cuda.synchronize()
    P.check_grad(P.to_host(xl, dtype), P.widen(x_rows, dtype), t_rows,
                 lse32.astype(np.float64), scale, dtype)


def check_case(x_np, t_np, dtype, reduction="mean", offset_elems=0, rows=None):
    out = run_all(x_np, t_np, dtype, reduction, offset_elems)
    M = x_np.shape[0]
    if rows is None:
        rows = np.arange(M)
    x64 = P.widen(x_np[rows], dtype)
    ref = oracle.ce_forward(x64, t_np[rows], reduction)
    tol = P.ROW_TOL[dtype]
    for key in ("rl_f", "rl_b"):
        P.check_rows(key, out[key].cpu().numpy(), ref["row_loss"], tol, rows)
    for key in ("lse_f", "lse_b"):
        P.check_lse(key, out[key].cpu().numpy(), ref["lse"], tol, rows)
    if reduction != "none":
        if len(rows) == M:
            P.check_loss(out["loss_f"].item(), ref["loss"], dtype, M)
            P.check_loss(out["loss_b"].item(), ref["loss"], dtype, M)
        # the reduction of the kernel's own row losses (any size)
        rl = out["rl_f"].cpu().numpy().astype(np.float64)
        own = rl.sum() / (M if reduction == "mean" else 1) if M else (
            float("nan") if reduction == "mean" else 0.0)
        for key in ("loss_f", "loss_b"):
            got = out[key].item()
            if np.isnan(own):
                assert np.isnan(got)
            else:
                assert abs(got - own) <= 1e-6 * max(1.0, abs(own)), (key, got, own)
    else:
        assert out["loss_f"] is None
    ridx = torch.from_numpy(rows).to(out["grad_b"].device)
    g = P.to_host(out["grad_b"][ridx], dtype)
    P.check_grad(g, x64, t_np[rows], ref["lse"], out["scale"], dtype)
    if M:
        check_backward_from_lse(x_np[rows], t_np[rows], ref["lse"], out["scale"], dtype,
                                offset_elems)
    return out


# ---------------------------------------------------------------------------
# Sweeps over V (tile/cluster boundaries, ragged tails) and M
# ---------------------------------------------------------------------------
V_SWEEP = [1, 2, 3, 7, 31, 32, 33, 127, 128, 129, 1000, 1024, 1025, 4095, 4096, 4097, 8191,
           16384, 16387, 32768, 32771, 50257, 65536, 65539, 100003, 131072, 128256, 256000,
           300007]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("V", V_SWEEP)
def test_sweep_vocab(dtype, V):
    assert V <= api().ce_max_vocab(dtype)
    M = max(2, min(300, (3 << 20) // V))
    sigma = {"f32": 1.0, "f16": 2.0, "bf16": 8.0}[dtype]
    x = synthetic.make_logits(M, V, dtype, sigma, seed=V)
    t = synthetic.make_targets(M, V, seed=V + 1)
    check_case(x, t, dtype)


@pytest.mark.parametrize("plan,dtype,V", [("3,32,1,2", "f32", 256), ("4,64,1,2", "bf16", 100),
                                          ("3,16,1,3", "f16", 999), ("4,32,1,2", "f32", 31)])
def test_sub_warp_row_groups_many_units(plan, dtype, V, monkeypatch):
    # 8 or 16 threads per row, many units per CTA and a ragged last unit
    monkeypatch.setenv("CE_KERNEL", "unit")
    monkeypatch.setenv("CE_PLAN", plan)
    M = 5003
    x = synthetic.make_logits(M, V, dtype, 3.0, seed=V + 21)
    t = synthetic.make_targets(M, V, seed=V + 22)
    t[17] = V  # one target out of range in the middle of a warp's rows
    a = api()
    assert a.ce_check_errors() == 0
    rows = np.unique(np.concatenate([P.sample_rows(M, 400), [16, 17, 18]]))
    check_case(x, t, dtype, "sum", rows=rows)
    assert a.ce_check_errors() == a.CE_ERR_TARGET_RANGE


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("V", [1, 7, 129, 4097, 50257, 131072, 300007])
def test_unit_kernel_in_every_mode(dtype, V, monkeypatch):
    # the forward (and the longest rows) default to the streaming kernel; the
    # unit kernel stays selectable and must agree with the oracle everywhere
    monkeypatch.setenv("CE_KERNEL", "unit")
    M = max(2, min(200, (2 << 20) // V))
    x = synthetic.make_logits(M, V, dtype, 2.0, seed=V + 7)
    t = synthetic.make_targets(M, V, seed=V + 8)
    check_case(x, t, dtype)


@pytest.mark.parametrize("dtype,V", [("f32", 9000), ("f32", 13000), ("bf16", 25013),
                                     ("f16", 27001), ("bf16", 16387), ("f32", 8193)])
def test_two_rows_per_unit_mid_rows(dtype, V):
    # rows of 32-54 KB in the writing modes run two rows per unit when there are
    # enough rows (M >= 2 x SMs): both rows of a unit, aligned or not
    M = 400
    x = synthetic.make_logits(M, V, dtype, 2.0, seed=V + 11)
    t = synthetic.make_targets(M, V, seed=V + 12)
    check_case(x, t, dtype, rows=P.sample_rows(M, 160))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 2, 3, 5, 151, 152, 153, 1000, 4099])
def test_sweep_rows(dtype, M):
    V = 777
    x = synthetic.make_logits(M, V, dtype, 3.0, seed=M)
    t = synthetic.make_targets(M, V, seed=M + 5)
    check_case(x, t, dtype)


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("dtype,V", [("f32", 4096), ("f16", 50257), ("bf16", 333)])
def test_reductions(reduction, dtype, V):
    M = 64
    x = synthetic.make_logits(M, V, dtype, 2.0, seed=3)
    t = synthetic.make_targets(M, V, seed=4)
    check_case(x, t, dtype, reduction)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("offset", [1, 3])
@pytest.mark.parametrize("V", [5, 1001, 4096, 50257])
def test_base_pointer_off_the_16_byte_grid(dtype, offset, V):
    M = 37
    x = synthetic.make_logits(M, V, dtype, 2.0, seed=11)
    t = synthetic.make_targets(M, V, seed=12)
    check_case(x, t, dtype, offset_elems=offset)


# ---------------------------------------------------------------------------
# Degenerate and special inputs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("V", [1, 17, 4096, 50257])
def test_uniform_rows_give_log_v(dtype, V):
    M = 8
    c = {"f32": 1234.5, "f16": -3.0, "bf16": 96.0}[dtype]
    x = np.full((M, V), c, dtype=np.float32)
    x = x if dtype == "f32" else (x.astype(np.float16) if dtype == "f16"
                                  else synthetic.f32_to_bf16_bits(x))
    t = synthetic.make_targets(M, V, seed=1)
    out = check_case(x, t, dtype)
    np.testing.assert_allclose(out["rl_f"].cpu().numpy(), math.log(V), atol=P.ROW_TOL[dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_negative_infinity_entries(dtype):
    M, V = 16, 4100
    x = synthetic.make_logits(M, V, "f32", 1.0, seed=5)
    x[:, ::3] = -np.inf
    t = synthetic.make_targets(M, V, seed=6)
    t = t - t % 3 + 1  # targets on finite entries (index = 1 mod 3 <= V - 1)
    xs = x if dtype == "f32" else synthetic.f32_to_bf16_bits(x)
    check_case(xs, t, dtype)


@pytest.mark.parametrize("kernel", ["unit", "stream"])
@pytest.mark.parametrize("dtype,V", [("f32", 3001), ("f16", 4099), ("bf16", 50257)])
def test_degenerate_rows(kernel, dtype, V, monkeypatch):
    # The method's degenerate rows, beside ordinary ones:
    #  * a row with no finite logit: the sum of exponentials is empty, so its
    #    lse is log 0 = -inf, and lse - x_t = -inf - (-inf) makes its loss and
    #    every gradient element NaN;
    #  * a row with one NaN logit: the NaN reaches the sum, so the row's lse,
    #    loss and gradient are NaN (the NaN-ignoring maxima must not hide it).
    # The other rows are unaffected and match the oracle; the mean is NaN.
    monkeypatch.setenv("CE_KERNEL", kernel)
    M = 6
    x = synthetic.make_logits(M, V, "f32", 1.0, seed=V + 41)
    x[1, :] = -np.inf
    x[3, V // 3] = np.nan
    t = synthetic.make_targets(M, V, seed=V + 42)
    xs = (x if dtype == "f32" else x.astype(np.float16) if dtype == "f16"
          else synthetic.f32_to_bf16_bits(x))
    out = run_all(xs, t, dtype, "mean")
    ok = np.array([0, 2, 4, 5])
    x64 = P.widen(xs[ok], dtype)
    ref = oracle.ce_forward(x64, t[ok], "sum")
    tol = P.ROW_TOL[dtype]
    for key in ("rl_f", "rl_b"):
        got = out[key].cpu().numpy()
        P.check_rows(key, got[ok], ref["row_loss"], tol)
        assert np.isnan(got[1]) and np.isnan(got[3]), (key, got)
    for key in ("lse_f", "lse_b"):
        got = out[key].cpu().numpy()
        P.check_lse(key, got[ok], ref["lse"], tol, None)
        assert got[1] == -np.inf and np.isnan(got[3]), (key, got)
    assert math.isnan(out["loss_f"].item()) and math.isnan(out["loss_b"].item())
    g = P.to_host(out["grad_b"], dtype)
    gw = oracle.to_f64(g, dtype)
    assert np.isnan(gw[1]).all() and np.isnan(gw[3]).all()
    P.check_grad(g[ok], x64, t[ok], ref["lse"], 1.0 / M, dtype)


def test_one_hot_dominant_and_large_offsets():
    M, V = 6, 3000
    x = np.zeros((M, V), dtype=np.float32)
    t = np.arange(M, dtype=np.int64) * 101
    x[np.arange(M), t] = 50.0
    x[3:] += np.float32(1e4)  # large shared offset: shift invariance
    out = check_case(x, t, "f32")
    assert np.all(out["rl_f"].cpu().numpy()[:3] < 1e-6)


def test_spiked_rows_fp16():
    w = synthetic.WORKLOADS["f16_8192x131072_spiked"]
    x = synthetic.make_logits(24, w.V, "f16", w.sigma, w.spike_prob, w.spike_value, seed=9)
    t = synthetic.make_targets(24, w.V, seed=10)
    check_case(x, t, "f16")


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_empty_batch(reduction):
    x = np.zeros((0, 10), dtype=np.float32)
    t = np.zeros(0, dtype=np.int64)
    a = api()
    loss, _, _ = a.ce_forward(torch.zeros((0, 10), device="cuda"), torch.from_numpy(t).cuda(),
                              reduction)
    loss2, _, _ = a.ce_fwd_bwd_inplace(torch.zeros((0, 10), device="cuda"),
                                       torch.from_numpy(t).cuda(), reduction)
    ref = oracle.ce_forward(x, t, reduction)["loss"]
    for L in (loss.item(), loss2.item()):
        assert (math.isnan(L) and math.isnan(ref)) or L == ref


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_out_of_range_targets(dtype):
    a = api()
    M, V = 12, 5000
    x = synthetic.make_logits(M, V, dtype, 1.0, seed=2)
    t = synthetic.make_targets(M, V, seed=3)
    t[2] = V
    t[7] = -4
    assert a.ce_check_errors() == 0
    check_case(x, t, dtype, "sum")
    assert a.ce_check_errors() == a.CE_ERR_TARGET_RANGE
    assert a.ce_check_errors() == 0  # the word was cleared


def test_bounded_wait_timeout_reports_and_recovers():
    a = api()
    assert a.ce_check_errors() == 0
    assert a.ce_selftest_wait_timeout(2000) == 0
    assert a.ce_check_errors() == a.CE_ERR_TIMEOUT
    assert a.ce_check_errors() == 0
    # the context is still usable
    x = synthetic.make_logits(4, 100, "f32", seed=1)
    check_case(x, synthetic.make_targets(4, 100), "f32")


def test_deterministic_repeat():
    a = api()
    M, V = 3000, 4096
    x = synthetic.make_logits(M, V, "f32", seed=21)
    t = torch.from_numpy(synthetic.make_targets(M, V, seed=22)).cuda()
    res = []
    for _ in range(3):
        xd = P.to_device(x, "f32")
        loss, rl, lse = a.ce_fwd_bwd_inplace(xd, t)
        res.append((loss.item(), rl.cpu().numpy(), lse.cpu().numpy(), xd.cpu().numpy()))
    for r in res[1:]:
        assert r[0] == res[0][0]
        for i in (1, 2, 3):
            assert np.array_equal(r[i], res[0][i])


def test_side_stream():
    x = synthetic.make_logits(100, 2049, "bf16", 8.0, seed=8)
    t = synthetic.make_targets(100, 2049, seed=9)
    s = torch.cuda.Stream()
    out = run_all(x, t, "bf16", stream=s)
    ref = oracle.ce_forward(P.widen(x, "bf16"), t, "mean")
    P.check_rows("rl", out["rl_b"].cpu().numpy(), ref["row_loss"], P.ROW_TOL["bf16"])


# CE_PLAN = "variant,R,CL,S"; variants: 0 = 256 threads x 8 register chunks,
# 1 = 512 x 4 register chunks, 2/3/4 = 128/256/512 threads re-reading shared memory
@pytest.mark.parametrize("plan,dtype,V", [
    ("0,2,1,3", "f32", 4096), ("1,2,1,3", "bf16", 1999), ("0,1,1,2", "f16", 4099),
    ("0,1,8,3", "f16", 131072), ("0,1,4,4", "bf16", 50257), ("1,1,8,2", "f32", 30000),
    ("1,16,1,6", "f32", 100), ("2,1,1,4", "f32", 4096), ("2,1,6,2", "bf16", 50257),
    ("4,4,1,3", "f16", 1000), ("4,1,2,2", "f32", 65539), ("3,8,1,2", "bf16", 7),
    # several rows in one warp: 16 or 8 threads per row
    ("3,16,1,2", "f32", 1000), ("3,32,1,2", "bf16", 333), ("4,64,1,2", "f16", 100),
    ("0,32,1,2", "f32", 200), ("1,32,1,3", "bf16", 500), ("2,16,1,4", "f16", 77),
])
def test_other_launch_shapes(plan, dtype, V, monkeypatch):
    monkeypatch.setenv("CE_KERNEL", "unit")  # the unit kernel in every mode
    monkeypatch.setenv("CE_PLAN", plan)
    M = max(2, min(64, (2 << 20) // V))
    x = synthetic.make_logits(M, V, dtype, 2.0, seed=V)
    t = synthetic.make_targets(M, V, seed=V + 2)
    check_case(x, t, dtype)


# ---------------------------------------------------------------------------
# The workloads at full size
# ---------------------------------------------------------------------------
def test_small_f32_256x1024_forward():
    x, t = synthetic.make_workload("small_f32_256x1024")
    a = api()
    loss, rl, lse = a.ce_forward(P.to_device(x, "f32"), torch.from_numpy(t).cuda(), "mean")
    ref = oracle.ce_forward(P.widen(x, "f32"), t, "mean")
    P.check_rows("row_loss", rl.cpu().numpy(), ref["row_loss"], P.ROW_TOL["f32"])
    P.check_rows("lse", lse.cpu().numpy(), ref["lse"], P.ROW_TOL["f32"])
    P.check_loss(loss.item(), ref["loss"], "f32", 256)


def test_f32_32768x4096_full():
    x, t = synthetic.make_workload("f32_32768x4096")
    rows = P.sample_rows(x.shape[0], 512)
    out = check_case(x, t, "f32", rows=rows)
    # the full-batch mean against the oracle, in row blocks
    x64_sum = 0.0
    for r0 in range(0, x.shape[0], 2048):
        f = oracle.ce_forward(x[r0:r0 + 2048].astype(np.float64), t[r0:r0 + 2048], "sum")
        x64_sum += f["loss"]
    P.check_loss(out["loss_b"].item(), x64_sum / x.shape[0], "f32", x.shape[0])
    P.check_loss(out["loss_f"].item(), x64_sum / x.shape[0], "f32", x.shape[0])


@pytest.mark.parametrize("name", ["f16_8192x131072_spiked", "bf16_16384x50257"])
def test_large_workloads_sampled(name):
    w = synthetic.WORKLOADS[name]
    x, t = synthetic.make_workload(w)
    rows = P.sample_rows(w.M, 128)
    out = check_case(x, t, w.dtype, rows=rows)
    # the deterministic mean over every row against the float64 oracle's mean
    # over every row (the per-row definition, reduced by a separate sum)
    ref = P.workload_full_loss(name)
    P.check_loss(out["loss_f"].item(), ref, w.dtype, w.M)
    P.check_loss(out["loss_b"].item(), ref, w.dtype, w.M)


@pytest.mark.parametrize("kernel", ["unit", "stream"])
@pytest.mark.parametrize("dtype,V", [("f32", 1000), ("bf16", 4099), ("f16", 50257),
                                     ("f32", 131072)])
def test_target_gradient_across_probability(kernel, dtype, V, monkeypatch):
    # rows whose target holds from almost none to almost all of the probability:
    # u = x_t - lse sweeps (-25, 0], across the switch at u = -1/2 between the
    # two forms of exp(u) - 1 used for the target's gradient
    monkeypatch.setenv("CE_KERNEL", kernel)
    M = 96
    x = synthetic.make_logits(M, V, "f32", 0.5, seed=V + 31)
    t = synthetic.make_targets(M, V, seed=V + 32)
    lift = np.linspace(-12.0, 12.0 + np.log(V), M)
    x[np.arange(M), t] = (np.max(x, axis=1) + lift).astype(np.float32)
    xs = (x if dtype == "f32" else x.astype(np.float16) if dtype == "f16"
          else synthetic.f32_to_bf16_bits(x))
    check_case(xs, t, dtype, "sum")


@pytest.mark.parametrize("plan", ["3,1,1,1", "2,2,1,1", "0,1,1,1", "3,1,2,1"])
def test_single_stage_pipeline_many_units_per_cta(plan, monkeypatch):
    # one stage: every refill waits for the previous store to be read out;
    # enough rows that each CTA runs many units
    monkeypatch.setenv("CE_KERNEL", "unit")
    monkeypatch.setenv("CE_PLAN", plan)
    M, V = 20000, 1000
    x = synthetic.make_logits(M, V, "f32", 2.0, seed=77)
    t = synthetic.make_targets(M, V, seed=78)
    check_case(x, t, "f32", rows=P.sample_rows(M, 400))
