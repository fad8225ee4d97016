"""ce_fwd_bwd_inplace_noalloc: the fused forward+backward for callers that
cannot allocate device memory (the library's reduction scratch is a fixed
array in its own device code).  Its results must match ce_fwd_bwd_inplace on
the same inputs, call after call, since every call reuses that one array, and
the float64 oracle within the parity tolerances.

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


# (kernel choice, launch shape): the default choice for the shape, or one forced
# through CE_KERNEL / CE_PLAN ("variant,R,CL,S"), so that the fixed scratch is
# handed to every kernel form that reduces: the unit kernel with several rows
# per unit and with one row per CTA, the unit kernel split over a cluster, and
# the warp-streaming kernel.
@pytest.mark.parametrize("dtype,M,V,reduction,kernel,plan", [
    ("f32", 4096, 4096, "mean", None, None),        # unit kernel, 4 rows per unit
    ("bf16", 300, 50257, "mean", None, None),       # unit kernel, one 100 KB row per CTA
    ("f16", 1000, 1001, "sum", None, None),         # misaligned rows, sum
    ("f16", 200, 131072, "mean", None, None),       # streaming kernel (256 KB rows)
    ("bf16", 64, 50257, "mean", "unit", "3,1,4,2"),  # unit kernel, clusters of 4 CTAs
    ("f32", 500, 3000, "sum", "stream", None),      # streaming kernel, a warp per row
])
def test_noalloc_matches_allocating_entry_point_twice(api, dtype, M, V, reduction, kernel, plan,
                                                      monkeypatch):
    if kernel is not None:
        monkeypatch.setenv("CE_KERNEL", kernel)
    if plan is not None:
        monkeypatch.setenv("CE_PLAN", plan)
    x = synthetic.make_logits(M, V, dtype, 4.0, seed=M + V)
    t = torch.from_numpy(synthetic.make_targets(M, V, seed=M)).cuda()
    dev = t.device
    # the float64 oracle on the same rows
    x64 = P.widen(x, dtype)
    ref = oracle.ce_forward(x64, t.cpu().numpy(), reduction)
    scale = 1.0 / M if reduction == "mean" else 1.0
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
        bound = (P.GRAD_TOL_F32 * scale if dtype == "f32"
                 else oracle.ulp(gb, dtype) + P.GRAD_ABS_EPS * scale)
        assert np.all(np.abs(ga - gb) <= bound), call
        # and against the oracle: row losses, lse, the reduced loss, the gradient
        P.check_rows("row_loss vs oracle", rl.cpu().numpy(), ref["row_loss"], tol)
        P.check_lse("lse vs oracle", lse.cpu().numpy(), ref["lse"], tol)
        P.check_loss(loss.item(), ref["loss"], dtype, M)
        P.check_grad(P.to_host(xa, dtype), x64, t.cpu().numpy(), ref["lse"], scale, dtype)
    assert api.ce_check_errors() == 0


def test_noalloc_without_reduction_and_rejects_bad_args(api, monkeypatch):
    monkeypatch.delenv("CE_KERNEL", raising=False)
    monkeypatch.delenv("CE_PLAN", raising=False)
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
