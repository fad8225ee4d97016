"""GPU parity of ce_softmax_forward (the fused row softmax) against the
float64 oracle.  Tolerance as for the gradient with scale 1: fp32 |p - p_ref|
<= 1e-5; 16-bit |p - RN(p_ref)| <= ulp(p_ref) + 4e-6."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from softmax_cross_entropy_online_gb300 import synthetic  # noqa: E402
from tests import parity as P  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_online_gb300 import api as a, build
    build.build()
    a.lib()
    return a


def check(p_storage, x_storage, dtype):
    p_ref = oracle.softmax_rows(P.widen(x_storage, dtype))
    p = oracle.to_f64(p_storage, dtype)
    if dtype == "f32":
        assert np.all(np.abs(p - p_ref) <= 1e-5)
    else:
        err = np.abs(p - oracle.round_to_format(p_ref, dtype))
        assert np.all(err <= oracle.ulp(p_ref, dtype) + 4e-6)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("V", [1, 7, 1000, 4096, 50257, 131072])
@pytest.mark.parametrize("inplace", [True, False])
def test_softmax_sweep(api, dtype, V, inplace):
    M = max(2, min(200, (2 << 20) // V))
    x = synthetic.make_logits(M, V, dtype, 3.0, seed=V)
    xd = P.to_device(x, dtype)
    probs, lse = api.ce_softmax_forward(xd, xd if inplace else None, lse=True)
    torch.cuda.synchronize()
    check(P.to_host(probs, dtype), x, dtype)
    ref_lse = oracle.logsumexp_rows(P.widen(x, dtype))
    P.check_lse("lse", lse.cpu().numpy(), ref_lse, P.ROW_TOL[dtype])
    if not inplace:  # the input is untouched
        assert np.array_equal(P.to_host(xd, dtype), x)
    assert api.ce_check_errors() == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_softmax_off_grid_base(api, dtype):
    M, V = 33, 1001
    x = synthetic.make_logits(M, V, dtype, 2.0, seed=4)
    xd = P.to_device(x, dtype, offset_elems=3)
    out = P.to_device(np.zeros_like(x), dtype, offset_elems=3)  # same 16-byte phase
    probs, _ = api.ce_softmax_forward(xd, out)
    torch.cuda.synchronize()
    check(P.to_host(probs, dtype), x, dtype)


def test_softmax_rejects_other_phase(api):
    x = torch.zeros((4, 9), dtype=torch.float16, device="cuda")
    buf = torch.zeros(4 * 9 + 1, dtype=torch.float16, device="cuda")
    with pytest.raises(api.CEError):
        api.ce_softmax_forward(x, buf[1:].view(4, 9))


@pytest.mark.parametrize("kernel", ["unit", "stream"])
@pytest.mark.parametrize("dtype,V", [("f32", 3001), ("bf16", 50257)])
def test_softmax_degenerate_rows(api, kernel, dtype, V, monkeypatch):
    # A row with no finite logit has an empty sum (lse = log 0 = -inf, and
    # 0/0 probabilities: NaN); a row with one NaN logit carries the NaN into
    # its sum, so its lse and every probability are NaN.  The other rows are
    # unaffected.
    monkeypatch.setenv("CE_KERNEL", kernel)
    M = 6
    x = synthetic.make_logits(M, V, "f32", 2.0, seed=V + 7)
    x[2, :] = -np.inf
    x[4, V // 2] = np.nan
    xs = x if dtype == "f32" else synthetic.f32_to_bf16_bits(x)
    xd = P.to_device(xs, dtype)
    probs, lse = api.ce_softmax_forward(xd, xd, lse=True)
    torch.cuda.synchronize()
    p = oracle.to_f64(P.to_host(probs, dtype), dtype)
    ok = np.array([0, 1, 3, 5])
    check(P.to_host(probs, dtype)[ok], xs[ok], dtype)
    assert np.isnan(p[2]).all() and np.isnan(p[4]).all()
    lse = lse.cpu().numpy()
    assert lse[2] == -np.inf and np.isnan(lse[4])
    P.check_lse("lse", lse[ok], oracle.logsumexp_rows(P.widen(xs[ok], dtype)), P.ROW_TOL[dtype])
