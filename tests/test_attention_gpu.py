"""GPU parity of the tensor-core blockwise attention forward against the
float64 oracle (oracle.attention_oracle.attention_forward) on the same bf16
inputs.

Tolerances, from the arithmetic of the kernel:
  * scores: exact bf16 products summed in fp32 by the tensor cores, so
    |S - S_ref| <= d_s = sm_scale * D * 2^-24 * max_j sum_d |q_d k_jd| per row
    (+ 2^-22 max_j |mask_ij| with an additive mask, which joins the unscaled
    score as fma(mask, 1/sm_scale, s));
    exp turns that into a relative error of at most d_s in each weight, on
    the numerator and on the normaliser alike;
  * P is rounded to bf16 (relative 2^-8: the unit roundoff of an 8-bit
    significand) before P V; the normaliser sums the
    unrounded fp32 weights; P V and the normaliser accumulate in fp32
    (relative T * 2^-24 at most);
so |O - O_ref| <= (2^-8 + 2 d_s + T 2^-24) (P_ref |V|) + 1e-6 elementwise, with
P_ref |V| the oracle run on |V|; rounded to bf16, the output moves by at most
2^-8 of the kernel's fp32 value, itself within that bound b of O_ref, so the bf16
output is held to b (1 + 2^-8) + 2^-8 |O_ref|; and
|lse - lse_ref| <= d_s + (T + 16) 2^-24 + 2^-22 |lse_ref| + 1e-6.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import attention_oracle as AO  # noqa: E402
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


def widen(bits):
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def check(out, lse, q, k, v, mask, sm_scale, heads=None, out16=False):
    """Compare kernel outputs with the oracle on the heads listed (all by
    default); q, k, v are bf16 bit patterns [B, NH, T, D]."""
    B, NH, T, D = q.shape
    q, k, v = (a.reshape(B * NH, T, D) for a in (q, k, v))
    out = out.reshape(B * NH, T, D)
    lse = None if lse is None else lse.reshape(B * NH, T)
    hs = range(B * NH) if heads is None else heads
    for h in hs:
        qh, kh, vh = widen(q[h]), widen(k[h]), widen(v[h])
        ref = AO.attention_forward(qh, kh, vh, mask, sm_scale)
        pv = AO.attention_forward(qh, kh, np.abs(vh), mask, sm_scale)["out"]
        d_s = sm_scale * D * 2.0 ** -24 * np.max(np.abs(qh) @ np.abs(kh).T, axis=1)
        if mask is not None:
            # the mask enters as fma(mask, 1/sm_scale, s): two more roundings
            fin = np.where(np.isfinite(mask), np.abs(mask), 0.0)
            d_s = d_s + 2.0 ** -22 * np.max(fin, axis=1)
        bound = (2.0 ** -8 + 2 * d_s[:, None] + T * 2.0 ** -24) * pv + 1e-6
        if out16:
            bound = bound * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(ref["out"])
        err = np.abs(out[h].astype(np.float64) - ref["out"])
        if not np.all(err <= bound):
            i, j = np.unravel_index(np.argmax(err / bound), err.shape)
            raise AssertionError(
                f"head {h} at ({i}, {j}): err {err[i, j]:.6g} > bound {bound[i, j]:.6g}; "
                f"got {out[h][i, j]!r}, ref {ref['out'][i, j]!r}, P|V| {pv[i, j]:.6g}, "
                f"d_s {d_s[i]:.3g}")
        if lse is not None:
            lb = d_s + (T + 16) * 2.0 ** -24 + 2.0 ** -22 * np.abs(ref["lse"]) + 1e-6
            le = np.abs(lse[h].astype(np.float64) - ref["lse"])
            assert np.all(le <= lb), f"head {h}: lse worst {np.max(le / lb):.3g} x bound"


def run(api, q, k, v, mask=None, causal=False, sm_scale=None, lse=True, out16=False):
    D = q.shape[-1]
    sm_scale = 1.0 / np.sqrt(D) if sm_scale is None else sm_scale
    mt = None if mask is None else torch.from_numpy(np.ascontiguousarray(mask, np.float32)).cuda()
    o, l = api.ce_attention_forward(bf16_dev(q), bf16_dev(k), bf16_dev(v), mt, causal=causal,
                                    sm_scale=sm_scale, lse=lse,
                                    out_dtype=torch.bfloat16 if out16 else torch.float32)
    torch.cuda.synchronize()
    assert api.ce_check_errors() == 0
    return o.float().cpu().numpy(), (None if l is None else l.cpu().numpy()), sm_scale


PAGE_T = [1, 2, 3, 4, 5, 8, 16, 32, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1023,
          1024]


@pytest.mark.parametrize("T", PAGE_T)
def test_page_sweep_causal_mask(api, T):
    # the page's correctness harness: B = 16, NH = 8, D = 64, an additive
    # causal mask, T straddling powers of two
    B, NH, D = 16, 8, 64
    q, k, v = synthetic.make_attention_inputs(B, NH, T, D, seed=T)
    mask = AO.causal_mask(T)
    o, l, sc = run(api, q, k, v, mask=mask)
    heads = None if T <= 129 else [0, 37, 90, 127]
    check(o, l, q, k, v, mask, sc, heads)
    # the causal flag (tiles above the diagonal skipped) gives the same bits:
    # a tile whose keys are all hidden adds exactly nothing
    o2, l2, _ = run(api, q, k, v, causal=True)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("T", [1, 100, 128, 129, 300, 640])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("out16", [False, True])
def test_shapes(api, D, T, causal, out16):
    B, NH = 2, 3
    q, k, v = synthetic.make_attention_inputs(B, NH, T, D, seed=1000 + T + D)
    o, l, sc = run(api, q, k, v, causal=causal, out16=out16)
    check(o, l, q, k, v, AO.causal_mask(T) if causal else None, sc, out16=out16)
    if out16:
        # the bf16 output is the fp32 output rounded to nearest even
        o32, l32, _ = run(api, q, k, v, causal=causal)
        r = torch.from_numpy(o32).to(torch.bfloat16).float().numpy()
        assert np.array_equal(o, r) and np.array_equal(l, l32)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("out16", [False, True])
def test_additive_mask_with_hidden_keys(api, causal, D, out16):
    B, NH, T = 1, 4, 333
    q, k, v = synthetic.make_attention_inputs(B, NH, T, D, seed=7)
    mask = synthetic.make_attention_mask(T, seed=8, sigma=2.0, hide_prob=0.3)
    o, l, sc = run(api, q, k, v, mask=mask, causal=causal, out16=out16)
    full = mask.astype(np.float64) + (AO.causal_mask(T) if causal else 0.0)
    check(o, l, q, k, v, full, sc, out16=out16)


def test_max_grows_in_every_key_tile(api):
    # scores rise along the key axis, so each new tile of 128 keys raises the
    # row max and the accumulator is rescaled after every tile
    B, NH, T, D = 1, 2, 768, 64
    q, k, v = synthetic.make_attention_inputs(B, NH, T, D, seed=11)
    qf = np.abs(widen(q)).astype(np.float32)
    ramp = np.linspace(0.0, 3.0, T, dtype=np.float32)[None, None, :, None]
    kf = (np.abs(widen(k)).astype(np.float32) * 0.1 + ramp)
    q, k = synthetic.f32_to_bf16_bits(qf), synthetic.f32_to_bf16_bits(kf)
    o, l, sc = run(api, q, k, v)
    check(o, l, q, k, v, None, sc)


def test_peaked_scores(api):
    # queries 4x larger: scores of several tens, nearly one-hot rows
    B, NH, T, D = 2, 2, 400, 128
    q, k, v = synthetic.make_attention_inputs(B, NH, T, D, seed=12, q_sigma=4.0)
    for causal in (False, True):
        o, l, sc = run(api, q, k, v, causal=causal)
        check(o, l, q, k, v, AO.causal_mask(T) if causal else None, sc)


def test_other_scale_and_no_lse(api):
    B, NH, T, D = 1, 3, 200, 64
    q, k, v = synthetic.make_attention_inputs(B, NH, T, D, seed=13)
    o, l, sc = run(api, q, k, v, sm_scale=0.37, lse=False)
    assert l is None
    check(o, None, q, k, v, None, sc)


def test_fully_hidden_row(api):
    # a query that sees no key: the definition's 0/0 -- NaN outputs, lse -inf;
    # every other row is unaffected
    B, NH, T, D = 1, 2, 150, 64
    q, k, v = synthetic.make_attention_inputs(B, NH, T, D, seed=14)
    mask = np.zeros((T, T), np.float32)
    mask[5, :] = -np.inf
    o, l, sc = run(api, q, k, v, mask=mask)
    assert np.all(np.isnan(o[:, :, 5])) and np.all(np.isneginf(l[:, :, 5]))
    keep = [i for i in range(T) if i != 5]
    ref_mask = mask[keep].astype(np.float64)
    for h in range(NH):
        ref = AO.attention_forward(widen(q)[0, h, keep], widen(k)[0, h], widen(v)[0, h],
                                   ref_mask, sc)
        np.testing.assert_allclose(o[0, h, keep], ref["out"], rtol=0, atol=2e-2)


def test_deterministic(api):
    B, NH, T, D = 4, 8, 513, 128
    q, k, v = synthetic.make_attention_inputs(B, NH, T, D, seed=15)
    o1, l1, _ = run(api, q, k, v, causal=True)
    o2, l2, _ = run(api, q, k, v, causal=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("out16", [True, False])
def test_page_benchmark_shape_sampled(api, out16):
    # the page's benchmark shape (B = 32, NH = 96, T = 512, D = 128, causal),
    # launched as the bench launches it (bf16 output, like q); sampled heads
    # against the oracle
    B, NH, T, D = 32, 96, 512, 128
    q, k, v = synthetic.make_attention_inputs(B, NH, T, D, seed=16)
    o, l, sc = run(api, q, k, v, causal=True, out16=out16)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    check(o, l, q, k, v, AO.causal_mask(T), sc, heads=[0, 1, 1500, 3071], out16=out16)


def test_side_stream(api):
    # launched on a stream other than the current one, the kernel orders itself on
    # that stream alone and gives the same bits
    B, NH, T, D = 2, 4, 700, 128
    q, k, v = synthetic.make_attention_inputs(B, NH, T, D, seed=17)
    qd, kd, vd = bf16_dev(q), bf16_dev(k), bf16_dev(v)
    o1, l1 = api.ce_attention_forward(qd, kd, vd, causal=True, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    o2, l2 = api.ce_attention_forward(qd, kd, vd, causal=True, out_dtype=torch.bfloat16,
                                      stream=side)
    side.synchronize()
    assert api.ce_check_errors(stream=side) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
