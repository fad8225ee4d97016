"""GPU parity of the tensor-core GEMM and of the fused linear + cross-entropy
against float64 references (numpy matmul for the GEMM, the oracle's
linear_ce for the fused path).

Tolerances.  h and W are exact bf16 values, so every product is exact in
fp32; the GEMM accumulates in fp32 on the tensor cores: |D - D_ref| <=
1e-5 * (|A| |B|^T) covers K up to several thousand terms at 2^-24 per step.
The gradients use G rounded to bf16 (relative error at most 2^-8, the unit
roundoff of an 8-bit significand) and fp32 accumulation:
|dH - dH_ref| <= 2^-8 (|G| |W|) and |dW - dW_ref| <= 2^-8 (|G|^T |h|),
elementwise, with G the float64 reference gradient: the bound is the worst case
of the rounding alone; the fp32 errors of the logits and of the accumulations
(up to 128256 terms) stay far below theirs, because the terms' rounding errors
do not all share one sign, and the float64 comparison shows it.  The loss follows the
16-bit-input rule (2e-3).
"""

import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from softmax_cross_entropy_online_gb300 import synthetic  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_online_gb300 import api as a, build
    build.build()
    a.lib()
    return a


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 300, 136), (1, 1, 8), (513, 1000, 4096),
                                   (1024, 2048, 1024), (130, 520, 72)])
def test_gemm_against_float64(api, M, N, K):
    rng = np.random.default_rng(M * 7 + N)
    A = synthetic.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    B = synthetic.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32))
    A64, B64 = oracle.decode_bf16(A), oracle.decode_bf16(B)
    ref = A64 @ B64.T
    bound = 1e-5 * (np.abs(A64) @ np.abs(B64).T) + 1e-30
    D = api.ce_gemm_bf16_tn(bf16_dev(A), bf16_dev(B))
    torch.cuda.synchronize()
    err = np.abs(D.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), f"worst {np.max(err / bound):.3g} x bound"
    # beta = 1 accumulates into D
    api.ce_gemm_bf16_tn(bf16_dev(A), bf16_dev(B), D, beta=1.0)
    torch.cuda.synchronize()
    err = np.abs(D.cpu().numpy().astype(np.float64) - 2 * ref)
    assert np.all(err <= 2 * bound)
    assert api.ce_check_errors() == 0


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, False), (True, True)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 300, 136), (1, 1, 8), (513, 1000, 777),
                                   (130, 520, 2049), (1024, 768, 72), (192, 320, 200),
                                   (640, 64, 1000)])
def test_gemm_operand_layouts_against_float64(api, a_mn, b_mn, M, N, K):
    # (M, N multiples of 64 load MN-major tiles with one 3-D box, others in
    # 64-wide 2-D boxes)
    # A read K-major ([M, K]) or MN-major (stored [K, M]); the same for B
    rng = np.random.default_rng(M * 13 + N + K)
    A = synthetic.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    B = synthetic.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32))
    A64, B64 = oracle.decode_bf16(A), oracle.decode_bf16(B)
    ref = A64 @ B64.T
    bound = 1e-5 * (np.abs(A64) @ np.abs(B64).T) + 1e-30

    def stored(X, mn):
        # rows padded to a multiple of 8 elements, as the strides require
        Xs = np.ascontiguousarray(X.T) if mn else X
        cols = Xs.shape[1]
        pad = (cols + 7) // 8 * 8
        buf = np.zeros((Xs.shape[0], pad), dtype=Xs.dtype)
        buf[:, :cols] = Xs
        return bf16_dev(buf)[:, :cols]

    Ad, Bd = stored(A, a_mn), stored(B, b_mn)
    D = api.ce_gemm_bf16(Ad, Bd, a_mn=a_mn, b_mn=b_mn)
    torch.cuda.synchronize()
    err = np.abs(D.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), f"worst {np.max(err / bound):.3g} x bound"
    api.ce_gemm_bf16(Ad, Bd, D, beta=1.0, a_mn=a_mn, b_mn=b_mn)
    torch.cuda.synchronize()
    err = np.abs(D.cpu().numpy().astype(np.float64) - 2 * ref)
    assert np.all(err <= 2 * bound)
    assert api.ce_check_errors() == 0


def check_linear(api, M, H, V, seed, workspace_bytes=None, schedule="lean"):
    h, W, t = synthetic.make_linear_ce_inputs(M, H, V, seed=seed)
    ws = None
    if workspace_bytes is not None:
        ws = torch.empty(workspace_bytes, dtype=torch.uint8, device="cuda")
    loss, dH, dW = api.linear_ce_fwd_bwd(bf16_dev(h), bf16_dev(W), torch.from_numpy(t).cuda(),
                                         workspace=ws, schedule=schedule)
    torch.cuda.synchronize()
    assert api.ce_check_errors() == 0
    h64, W64 = oracle.decode_bf16(h), oracle.decode_bf16(W)
    ref = oracle.linear_ce(h64, W64, t, "mean")
    assert abs(loss.item() - ref["loss"]) <= 2e-3
    G = np.abs(ref["grad"])
    bH = 2.0**-8 * (G @ np.abs(W64)) + 1e-30
    eH = np.abs(dH.cpu().numpy().astype(np.float64) - ref["dH"])
    assert np.all(eH <= bH), f"dH worst {np.max(eH / bH):.3g} x bound"
    bW = 2.0**-8 * (G.T @ np.abs(h64)) + 1e-30
    eW = np.abs(dW.cpu().numpy().astype(np.float64) - ref["dW"])
    assert np.all(eW <= bW), f"dW worst {np.max(eW / bW):.3g} x bound"


@pytest.mark.parametrize("schedule", ["lean", "fused"])
@pytest.mark.parametrize("M,H,V", [(300, 256, 1000), (257, 64, 777), (128, 4096, 2048),
                                   (1, 8, 3), (64, 512, 50257)])
def test_linear_ce_against_oracle(api, M, H, V, schedule):
    check_linear(api, M, H, V, seed=M + H + V, schedule=schedule)


@pytest.mark.parametrize("M,H,V", [(5000, 256, 3001), (4224, 64, 1027), (2049, 128, 256)])
def test_linear_ce_fused_chunks_against_oracle(api, M, H, V):
    # several 2048-row chunks with the fused workspace: each chunk's gradient
    # rows are formed by the next chunk's GEMM epilogue, the last chunk's by the
    # standalone pass; V off the 4- and 256-column grids
    check_linear(api, M, H, V, seed=M + V, schedule="fused")


@pytest.mark.parametrize("M,H,V", [(5000, 256, 3001), (6000, 64, 1027), (2561, 128, 256),
                                   (3000, 4096, 300)])
def test_linear_ce_lean_chunks_against_oracle(api, M, H, V):
    # several row chunks with the default (lean) workspace: each chunk's pairs,
    # merged row constants and recomputed bf16 G, dW accumulated across the
    # chunks; V off the 4- and 256-column grids; H = 4096 takes 16 dH column tiles
    check_linear(api, M, H, V, seed=M + V + 1)


@pytest.mark.parametrize("workspace", ["lean", "fused", "lean_128_row_chunks"])
def test_linear_ce_out_of_range_targets(api, workspace):
    # targets outside [0, V) in the first and the last row chunk (in the fused
    # schedule the last one's gradient rows come from the standalone pass): those
    # rows' losses are NaN, so the mean is NaN, their gradient rows drop the
    # one-hot term, and the device error word is set; every other row is unaffected
    M, H, V = 4500, 64, 1003
    h, W, t = synthetic.make_linear_ce_inputs(M, H, V, seed=17)
    t[7] = V
    t[4400] = -2
    ws = None
    if workspace == "lean_128_row_chunks":
        ws = torch.empty(api.linear_ce_workspace_size(128, H, V) + 4 * M + 4096,
                         dtype=torch.uint8, device="cuda")
    assert api.ce_check_errors() == 0
    loss, dH, dW = api.linear_ce_fwd_bwd(bf16_dev(h), bf16_dev(W), torch.from_numpy(t).cuda(),
                                         workspace=ws,
                                         schedule="fused" if workspace == "fused" else "lean")
    torch.cuda.synchronize()
    assert api.ce_check_errors() == api.CE_ERR_TARGET_RANGE
    assert api.ce_check_errors() == 0
    h64, W64 = oracle.decode_bf16(h), oracle.decode_bf16(W)
    ref = oracle.linear_ce(h64, W64, t, "mean")
    assert np.isnan(ref["loss"]) and np.isnan(loss.item())
    G = np.abs(ref["grad"])
    eH = np.abs(dH.cpu().numpy().astype(np.float64) - ref["dH"])
    assert np.all(eH <= 2.0**-8 * (G @ np.abs(W64)) + 1e-30)
    eW = np.abs(dW.cpu().numpy().astype(np.float64) - ref["dW"])
    assert np.all(eW <= 2.0**-8 * (G.T @ np.abs(h64)) + 1e-30)


def test_linear_ce_in_row_chunks(api):
    # a workspace with room for 128 rows at a time: the lean schedule in chunks of 128
    M, H, V = 700, 128, 1500
    ws = api.linear_ce_workspace_size(128, H, V) + 4 * M + 4096
    check_linear(api, M, H, V, seed=5, workspace_bytes=ws)


def test_linear_ce_rejects_bad_layouts(api):
    h = torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda")  # H not a multiple of 8
    W = torch.zeros((5, 12), dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(api.CEError):
        api.linear_ce_fwd_bwd(h, W, t)


@pytest.mark.parametrize("schedule", ["lean", "fused"])
def test_linear_ce_full_width_sampled(api, schedule):
    # the bench shapes' H and V at 512 rows: all of loss and dH, sampled rows of dW
    M, H, V = 512, 4096, 128256
    h, W, t = synthetic.make_linear_ce_inputs(M, H, V, seed=0)
    loss, dH, dW = api.linear_ce_fwd_bwd(bf16_dev(h), bf16_dev(W), torch.from_numpy(t).cuda(),
                                         schedule=schedule)
    torch.cuda.synchronize()
    assert api.ce_check_errors() == 0
    h64, W64 = oracle.decode_bf16(h), oracle.decode_bf16(W)
    logits = h64 @ W64.T
    f = oracle.ce_fwd_bwd(logits, t, "mean")
    assert abs(loss.item() - f["loss"]) <= 2e-3
    G = f["grad"]
    eH = np.abs(dH.cpu().numpy().astype(np.float64) - G @ W64)
    assert np.all(eH <= 2.0**-8 * (np.abs(G) @ np.abs(W64)) + 1e-30)
    rng = np.random.default_rng(1)
    vs = np.unique(np.concatenate([t[:64], rng.choice(V, 192, replace=False), [0, V - 1]]))
    dW_ref = G[:, vs].T @ h64
    eW = np.abs(dW[torch.from_numpy(vs).cuda()].cpu().numpy().astype(np.float64) - dW_ref)
    assert np.all(eW <= 2.0**-8 * (np.abs(G[:, vs]).T @ np.abs(h64)) + 1e-30)


@functools.lru_cache(maxsize=1)
def bench_size_reference():
    """float64 loss, and rows of dH and dW, of the bench workload (h [8192, 4096],
    W [128256, 4096], seed 0), its logits formed 512 rows at a time: the rows
    straddle every chunk border of both schedules (2048-row chunks in the fused
    one; 2432 rows in the lean one on 152 SMs, where 19 x 16 dH tiles fill two
    waves)."""
    M, H, V = 8192, 4096, 128256
    h, W, t = synthetic.make_linear_ce_inputs(M, H, V, seed=0)
    h64, W64 = oracle.decode_bf16(h), oracle.decode_bf16(W)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([rng.choice(M, 16, replace=False),
                                     [0, 2047, 2048, 2431, 2432, 4095, 4096, 4863, 4864, 6143,
                                      6144, 7295, 7296, M - 1]]))
    vs = np.unique(np.concatenate([t[:32], rng.choice(V, 32, replace=False), [0, V - 1]]))
    total = 0.0
    dW_ref = np.zeros((len(vs), H))
    dW_bnd = np.zeros((len(vs), H))
    dH_ref, dH_bnd = {}, {}
    for b0 in range(0, M, 512):
        hb = h64[b0:b0 + 512]
        x = hb @ W64.T
        f = oracle.ce_forward(x, t[b0:b0 + 512], "sum")
        total += f["loss"]
        G = oracle.ce_grad(x, t[b0:b0 + 512], f["lse"], 1.0 / M)
        dW_ref += G[:, vs].T @ hb
        dW_bnd += np.abs(G[:, vs]).T @ np.abs(hb)
        for r in rows[(rows >= b0) & (rows < b0 + 512)]:
            dH_ref[r] = G[r - b0] @ W64
            dH_bnd[r] = np.abs(G[r - b0]) @ np.abs(W64)
    return (h, W, t), rows, vs, total / M, dH_ref, dH_bnd, dW_ref, dW_bnd


@pytest.mark.parametrize("schedule", ["lean", "fused"])
def test_linear_ce_bench_size_sampled(api, schedule):
    # the bench workload itself through the same call, in both schedules (dW
    # accumulated across the chunks in the lean one): the loss in full, and rows
    # of dH and dW, against the float64 reference
    (h, W, t), rows, vs, loss_ref, dH_ref, dH_bnd, dW_ref, dW_bnd = bench_size_reference()
    loss, dH, dW = api.linear_ce_fwd_bwd(bf16_dev(h), bf16_dev(W), torch.from_numpy(t).cuda(),
                                         schedule=schedule)
    torch.cuda.synchronize()
    assert api.ce_check_errors() == 0
    assert abs(loss.item() - loss_ref) <= 2e-3
    got_H = dH[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    for k, r in enumerate(rows):
        e = np.abs(got_H[k] - dH_ref[r])
        assert np.all(e <= 2.0**-8 * dH_bnd[r] + 1e-30), f"dH row {r}: worst {np.max(e / (2.0**-8 * dH_bnd[r] + 1e-30)):.3g} x bound"
    got_W = dW[torch.from_numpy(vs).cuda()].cpu().numpy().astype(np.float64)
    eW = np.abs(got_W - dW_ref)
    assert np.all(eW <= 2.0**-8 * dW_bnd + 1e-30), f"dW worst {np.max(eW / (2.0**-8 * dW_bnd + 1e-30)):.3g} x bound"
