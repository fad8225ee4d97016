"""ce_fwd_bwd_inplace_noalloc: the fused forward+backward for callers that
cannot allocate device memory (the library's reduction scratch is a fixed
array in its own device code).  Its results must match ce_fwd_bwd_inplace on
the same inputs, call after call, since every call reuses that one array.

This file is collected last on purpose: a failure here leaves every other
test already run.  It passes alone in a fresh process and after the others.
"""

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")

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


@pytest.mark.parametrize("dtype,M,V,reduction", [
    ("f32", 4096, 4096, "mean"),       # one CTA per row group
    ("bf16", 300, 50257, "mean"),      # rows split over a cluster
    ("f16", 1000, 1001, "sum"),        # misaligned rows, sum
])
def test_noalloc_matches_allocating_entry_point_twice(api, dtype, M, V, reduction):
    x = synthetic.make_logits(M, V, dtype, 4.0, seed=M + V)
    t = torch.from_numpy(synthetic.make_targets(M, V, seed=M)).cuda()
    dev = t.device
    # reference: the allocating entry point
    xr = P.to_device(x, dtype)
    loss_r, rl_r, lse_r = api.ce_fwd_bwd_inplace(xr, t, reduction)
    g_r = P.to_host(xr, dtype)
    # two calls in a row into caller-owned outputs (the scratch is reused)
    for call in range(2):
        xa = P.to_device(x, dtype)
        loss = torch.full((), float("nan"), dtype=torch.float32, device=dev)
        rl = torch.empty(M, dtype=torch.float32, device=dev)
        lse = torch.empty(M, dtype=torch.float32, device=dev)
        api.ce_fwd_bwd_inplace_noalloc(xa, t, reduction, loss=loss, row_loss=rl, lse=lse)
        torch.cuda.synchronize()
        tol = P.ROW_TOL[dtype]
        assert abs(loss.item() - loss_r.item()) <= (
            P.LOSS_REL_TOL_F32 * abs(loss_r.item()) if dtype == "f32" else tol), call
        P.check_rows("row_loss", rl.cpu().numpy(), rl_r.cpu().numpy().astype(np.float64), tol)
        P.check_rows("lse", lse.cpu().numpy(), lse_r.cpu().numpy().astype(np.float64), tol)
        ga = oracle.to_f64(P.to_host(xa, dtype), dtype)
        gb = oracle.to_f64(g_r, dtype)
        scale = 1.0 / M if reduction == "mean" else 1.0
        bound = (P.GRAD_TOL_F32 * scale if dtype == "f32"
                 else oracle.ulp(gb, dtype) + P.GRAD_ABS_EPS * scale)
        assert np.all(np.abs(ga - gb) <= bound), call
    assert api.ce_check_errors() == 0


def test_noalloc_without_reduction_and_rejects_bad_args(api):
    M, V = 64, 777
    x = synthetic.make_logits(M, V, "f32", seed=5)
    t = torch.from_numpy(synthetic.make_targets(M, V, seed=6)).cuda()
    xa = P.to_device(x, "f32")
    rl = torch.empty(M, dtype=torch.float32, device="cuda")
    api.ce_fwd_bwd_inplace_noalloc(xa, t, "none", row_loss=rl)
    xr = P.to_device(x, "f32")
    _, rl_r, _ = api.ce_fwd_bwd_inplace(xr, t, "none")
    torch.cuda.synchronize()
    P.check_rows("row_loss", rl.cpu().numpy(), rl_r.cpu().numpy().astype(np.float64), 1e-4)
    st = api.lib().ce_fwd_bwd_inplace_noalloc(xa.data_ptr(), t.data_ptr(), M, 0, 0, 0,
                                              None, None, None, None)
    assert st == api.CE_ERR_INVALID_ARG
