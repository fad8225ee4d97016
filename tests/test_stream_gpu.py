"""GPU parity of the warp-streaming row kernel (ce_stream.cuh) against the
float64 oracle: the same checks as the unit-kernel tests (forward, fused
fwd+bwd, backward from a stored lse, softmax), with the streaming kernel
forced through CE_KERNEL=stream and its launch shape through
CE_SPLAN="warps per CTA, warps per row, ring slots, segment bytes"."""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from softmax_cross_entropy_online_gb300 import synthetic  # noqa: E402
from tests import parity as P  # noqa: E402
from tests.test_parity_gpu import check_case  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_online_gb300 import api, build
    build.build()
    api.lib()
    yield


@pytest.fixture(autouse=True)
def _stream_kernel(monkeypatch):
    monkeypatch.setenv("CE_KERNEL", "stream")
    monkeypatch.delenv("CE_SPLAN", raising=False)
    yield


def api():
    from softmax_cross_entropy_online_gb300 import api as a
    return a


V_SWEEP = [1, 2, 3, 7, 31, 33, 129, 1000, 1025, 4096, 4097, 16387, 50257, 65539, 131072, 128256]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("V", V_SWEEP)
def test_stream_sweep_vocab(dtype, V):
    M = max(2, min(300, (3 << 20) // V))
    sigma = {"f32": 1.0, "f16": 2.0, "bf16": 8.0}[dtype]
    x = synthetic.make_logits(M, V, dtype, sigma, seed=V + 100)
    t = synthetic.make_targets(M, V, seed=V + 101)
    check_case(x, t, dtype)
    assert api().ce_check_errors() == 0


@pytest.mark.parametrize("M", [1, 2, 151, 152, 153, 2433, 5000])
def test_stream_sweep_rows(M):
    V = 777
    x = synthetic.make_logits(M, V, "bf16", 3.0, seed=M)
    t = synthetic.make_targets(M, V, seed=M + 5)
    check_case(x, t, "bf16", rows=P.sample_rows(M, 600))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("offset", [1, 3])
@pytest.mark.parametrize("V", [5, 1001, 4096, 50257])
def test_stream_base_off_the_16_byte_grid(dtype, offset, V):
    M = 37
    x = synthetic.make_logits(M, V, dtype, 2.0, seed=11)
    t = synthetic.make_targets(M, V, seed=12)
    check_case(x, t, dtype, offset_elems=offset)


# warps per CTA, warps per row, slots, segment bytes: one warp per row and
# whole-CTA rows, single-slot rings, segments smaller than a row and larger
@pytest.mark.parametrize("splan,dtype,V", [
    ("16,1,3,4096", "f32", 4096), ("8,2,4,2048", "bf16", 1999), ("12,4,3,4096", "f16", 50257),
    ("16,16,3,4096", "f16", 131072), ("4,4,2,512", "f32", 3001), ("16,1,1,512", "bf16", 4099),
    ("9,1,5,1024", "f32", 100), ("16,8,2,8192", "bf16", 50257), ("2,2,8,512", "f16", 17),
    ("16,16,1,512", "f32", 30000), ("8,8,3,1024", "bf16", 7), ("16,1,8,64", "f32", 9),
    ("16,1,8,16", "bf16", 3), ("4,1,8,32", "f16", 30),
])
def test_stream_launch_shapes(splan, dtype, V, monkeypatch):
    monkeypatch.setenv("CE_SPLAN", splan)
    M = max(2, min(64, (2 << 20) // V))
    x = synthetic.make_logits(M, V, dtype, 2.0, seed=V)
    t = synthetic.make_targets(M, V, seed=V + 2)
    check_case(x, t, dtype)


# resident rows (fifth field 1): every lane holds its chunks of the row in
# registers; fused fwd+bwd and softmax, across piece sizes, alignments and
# the partial head / tail chunks
@pytest.mark.parametrize("splan,dtype,V,offset", [
    ("16,16,3,4096,1", "bf16", 50257, 0), ("16,16,3,4096,1", "f16", 50257, 3),
    ("16,4,3,4096,1", "f32", 4096, 0), ("16,2,3,4096,1", "f32", 4096, 0),
    ("16,2,2,4096,1", "f32", 4097, 1), ("16,1,2,4096,1", "bf16", 1999, 5),
    ("16,1,3,4096,1", "f16", 7, 1), ("8,8,3,4096,1", "bf16", 30011, 0),
    ("16,16,2,4096,1", "f32", 32768, 0), ("16,4,3,4096,1", "bf16", 16387, 2),
])
def test_stream_resident_rows(splan, dtype, V, offset, monkeypatch):
    monkeypatch.setenv("CE_SPLAN", splan)
    M = max(2, min(80, (2 << 20) // V))
    x = synthetic.make_logits(M, V, dtype, 3.0, seed=V + 3)
    t = synthetic.make_targets(M, V, seed=V + 4)
    check_case(x, t, dtype, offset_elems=offset)
    xd = P.to_device(x, dtype, offset_elems=offset)
    probs, _ = api().ce_softmax_forward(xd, xd)
    torch.cuda.synchronize()
    p_ref = oracle.softmax_rows(P.widen(x, dtype))
    pg = oracle.to_f64(P.to_host(probs, dtype), dtype)
    if dtype == "f32":
        assert np.all(np.abs(pg - p_ref) <= 1e-5)
    else:
        err = np.abs(pg - oracle.round_to_format(p_ref, dtype))
        assert np.all(err <= oracle.ulp(p_ref, dtype) + 4e-6)


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_stream_reductions(reduction):
    x = synthetic.make_logits(64, 4096, "f32", 2.0, seed=3)
    t = synthetic.make_targets(64, 4096, seed=4)
    check_case(x, t, "f32", reduction)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("V", [1, 17, 4096, 50257])
def test_stream_uniform_rows_give_log_v(dtype, V):
    M = 8
    c = {"f32": 1234.5, "f16": -3.0, "bf16": 96.0}[dtype]
    x = np.full((M, V), c, dtype=np.float32)
    x = x if dtype == "f32" else (x.astype(np.float16) if dtype == "f16"
                                  else synthetic.f32_to_bf16_bits(x))
    t = synthetic.make_targets(M, V, seed=1)
    out = check_case(x, t, dtype)
    np.testing.assert_allclose(out["rl_f"].cpu().numpy(), math.log(V), atol=P.ROW_TOL[dtype])


@pytest.mark.parametrize("splan", ["16,1,3,4096", "16,4,2,512"])
def test_stream_negative_infinity_entries(splan, monkeypatch):
    monkeypatch.setenv("CE_SPLAN", splan)
    M, V = 16, 4100
    x = synthetic.make_logits(M, V, "f32", 1.0, seed=5)
    x[:, ::3] = -np.inf
    x[3, : V // 2] = -np.inf  # a whole segment of -inf before the finite values
    t = synthetic.make_targets(M, V, seed=6)
    t = t - t % 3 + 1
    t[3] = 2050  # finite: past the -inf half and not a multiple of 3
    check_case(x, t, "f32")
    check_case(synthetic.f32_to_bf16_bits(x), t, "bf16")


def test_stream_one_hot_dominant_and_large_offsets():
    M, V = 6, 3000
    x = np.zeros((M, V), dtype=np.float32)
    t = np.arange(M, dtype=np.int64) * 101
    x[np.arange(M), t] = 50.0
    x[3:] += np.float32(1e4)
    out = check_case(x, t, "f32")
    assert np.all(out["rl_f"].cpu().numpy()[:3] < 1e-6)


def test_stream_rising_rows_rescale_every_segment(monkeypatch):
    # the running max grows in every segment: every online rescale is taken
    monkeypatch.setenv("CE_SPLAN", "4,1,2,512")
    M, V = 8, 9000
    x = (np.arange(V, dtype=np.float32)[None, :] * np.float32(0.01)
         + synthetic.make_logits(M, V, "f32", 0.1, seed=3))
    t = synthetic.make_targets(M, V, seed=4)
    check_case(x.astype(np.float32), t, "f32")


def test_stream_spiked_rows_fp16():
    w = synthetic.WORKLOADS["f16_8192x131072_spiked"]
    x = synthetic.make_logits(24, w.V, "f16", w.sigma, w.spike_prob, w.spike_value, seed=9)
    t = synthetic.make_targets(24, w.V, seed=10)
    check_case(x, t, "f16")


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_stream_empty_batch(reduction):
    t = np.zeros(0, dtype=np.int64)
    a = api()
    loss, _, _ = a.ce_forward(torch.zeros((0, 10), device="cuda"), torch.from_numpy(t).cuda(),
                              reduction)
    loss2, _, _ = a.ce_fwd_bwd_inplace(torch.zeros((0, 10), device="cuda"),
                                       torch.from_numpy(t).cuda(), reduction)
    ref = oracle.ce_forward(np.zeros((0, 10)), t, reduction)["loss"]
    for L in (loss.item(), loss2.item()):
        assert (math.isnan(L) and math.isnan(ref)) or L == ref


def test_stream_out_of_range_targets():
    a = api()
    M, V = 12, 5000
    x = synthetic.make_logits(M, V, "f16", 1.0, seed=2)
    t = synthetic.make_targets(M, V, seed=3)
    t[2] = V
    t[7] = -4
    assert a.ce_check_errors() == 0
    check_case(x, t, "f16", "sum")
    assert a.ce_check_errors() == a.CE_ERR_TARGET_RANGE
    assert a.ce_check_errors() == 0


def test_stream_deterministic_repeat():
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


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("inplace", [True, False])
@pytest.mark.parametrize("V", [7, 4096, 50257])
def test_stream_softmax(dtype, inplace, V):
    a = api()
    M = max(2, min(200, (2 << 20) // V))
    x = synthetic.make_logits(M, V, dtype, 3.0, seed=V)
    # off the 16-byte grid in place (out of place, probs must share the input's phase)
    xd = P.to_device(x, dtype, offset_elems=3 if (V == 7 and inplace) else 0)
    probs, lse = a.ce_softmax_forward(xd, xd if inplace else None, lse=True)
    torch.cuda.synchronize()
    p_ref = oracle.softmax_rows(P.widen(x, dtype))
    p = oracle.to_f64(P.to_host(probs, dtype), dtype)
    if dtype == "f32":
        assert np.all(np.abs(p - p_ref) <= 1e-5)
    else:
        err = np.abs(p - oracle.round_to_format(p_ref, dtype))
        assert np.all(err <= oracle.ulp(p_ref, dtype) + 4e-6)
    P.check_lse("lse", lse.cpu().numpy(), oracle.logsumexp_rows(P.widen(x, dtype)),
                P.ROW_TOL[dtype])
    if not inplace:
        assert np.array_equal(P.to_host(xd, dtype), x)
    assert a.ce_check_errors() == 0


@pytest.mark.parametrize("name", ["f32_32768x4096", "f16_8192x131072_spiked",
                                  "bf16_16384x50257"])
def test_stream_workloads_sampled(name):
    w = synthetic.WORKLOADS[name]
    x, t = synthetic.make_workload(w)
    out = check_case(x, t, w.dtype, rows=P.sample_rows(w.M, 128))
    # the mean over every row against the float64 oracle's
    ref = P.workload_full_loss(name)
    P.check_loss(out["loss_f"].item(), ref, w.dtype, w.M)
    P.check_loss(out["loss_b"].item(), ref, w.dtype, w.M)
