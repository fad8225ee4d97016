"""The C ABI without a GPU: the library builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""

import ctypes
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

HEADER_DIR = os.path.join(ROOT, "include")


def _declared_functions():
    names = []
    for h in sorted(os.listdir(HEADER_DIR)):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\*?\s+(\w+)\s*\(", text, re.M):
            if m.group(1) not in ("if", "return"):
                names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def cdll():
    from softmax_cross_entropy_online_gb300 import api, build
    build.build()
    return api.lib()


def test_header_declares_the_boundary():
    names = set(_declared_functions())
    for required in ("ce_forward", "ce_fwd_bwd_inplace", "ce_backward_from_lse",
                     "ce_check_errors", "ce_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(cdll):
    from softmax_cross_entropy_online_gb300 import build
    names = _declared_functions()
    assert names
    exported = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH],
                              capture_output=True, text=True, check=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", exported, re.M), f"{n} not exported"
        assert hasattr(cdll, n)


def test_binding_covers_every_declared_symbol():
    from softmax_cross_entropy_online_gb300 import api
    assert set(_declared_functions()) == set(api.SIGNATURES)


def test_status_strings(cdll):
    from softmax_cross_entropy_online_gb300 import api
    names = [api.status_string(i) for i in range(6)]
    assert names == ["CE_OK", "CE_ERR_INVALID_ARG", "CE_ERR_UNSUPPORTED", "CE_ERR_TARGET_RANGE",
                     "CE_ERR_CUDA", "CE_ERR_TIMEOUT"]
    assert api.status_string(99) == "CE_ERR_UNKNOWN"


def test_max_vocab(cdll):
    assert cdll.ce_max_vocab(0) * 4 == cdll.ce_max_vocab(1) * 2 == cdll.ce_max_vocab(2) * 2
    # 8 CTAs x one 200 KB stage of 16-byte chunks, less two chunks of slack for a
    # misaligned row
    chunks = 8 * (200 * 1024 // 16) - 2
    assert cdll.ce_max_vocab(1) == chunks * 8 and cdll.ce_max_vocab(0) == chunks * 4
    assert cdll.ce_max_vocab(7) == 0


@pytest.mark.parametrize("args", [
    # (logits, targets, M, V, dtype, red, loss, row_loss, lse)
    (16, 16, -1, 4, 0, 0, 16, None, None),      # M < 0
    (16, 16, 4, 0, 0, 0, 16, None, None),       # V < 1
    (16, 16, 4, 4, 3, 0, 16, None, None),       # bad dtype
    (16, 16, 4, 4, 0, 5, 16, None, None),       # bad reduction
    (None, 16, 4, 4, 0, 0, 16, None, None),     # null logits
    (16, None, 4, 4, 0, 0, 16, None, None),     # null targets
    (18, 16, 4, 4, 0, 0, 16, None, None),       # fp32 logits not 4-byte aligned
    (17, 16, 4, 4, 1, 0, 16, None, None),       # fp16 logits not 2-byte aligned
    (16, 12, 4, 4, 0, 0, 16, None, None),       # targets not 8-byte aligned
    (16, 16, 4, 4, 0, 0, 18, None, None),       # loss not 4-byte aligned
    (16, 16, 4, 4, 0, 0, 16, 2, None),          # row_loss misaligned
    (16, 16, 1 << 40, 1 << 30, 0, 0, 16, None, None),  # M*V*4 overflows
])
def test_host_validation_rejects(cdll, args):
    for fn in (cdll.ce_forward, cdll.ce_fwd_bwd_inplace):
        assert fn(*args, None) == 1  # CE_ERR_INVALID_ARG, returned before any CUDA call


def test_host_validation_backward(cdll):
    assert cdll.ce_backward_from_lse(16, 16, None, 4, 4, 0, 1.0, None) == 1  # null lse
    assert cdll.ce_backward_from_lse(16, 16, 16, 4, 0, 0, 1.0, None) == 1    # V = 0
    assert cdll.ce_selftest_wait_timeout(None, 0) == 1
    assert cdll.ce_selftest_wait_timeout(None, 2000000) == 1


def test_empty_problem_without_loss_is_a_no_op(cdll):
    # M == 0 with nothing to write returns before touching the device
    assert cdll.ce_forward(None, None, 0, 5, 0, 2, None, None, None, None) == 0
    assert cdll.ce_fwd_bwd_inplace(None, None, 0, 5, 2, 0, None, None, None, None) == 0


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "softmax_cross_entropy_online_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", text, re.M), f
                assert "ce_oracle" not in text, f


@pytest.mark.parametrize("args, status", [
    # (q, k, v, mask, causal, B, NH, T, D, sm_scale, out, out_dtype, lse) -> status,
    # before any CUDA call
    ((16, 16, 16, None, 2, 1, 1, 8, 64, 0.125, 16, 0, None), 1),           # causal not 0/1
    ((16, 16, 16, None, 0, -1, 1, 8, 64, 0.125, 16, 0, None), 1),          # B < 0
    ((16, 16, 16, None, 0, 1, 1, -8, 64, 0.125, 16, 0, None), 1),          # T < 0
    ((16, 16, 16, None, 0, 1, 1, 8, 64, float("nan"), 16, 0, None), 1),    # sm_scale not finite
    ((16, 16, 16, None, 0, 1, 1, 8, 64, float("inf"), 16, 0, None), 1),
    ((16, 16, 16, None, 0, 1, 1, 8, 64, 0.0, 16, 0, None), 1),             # sm_scale not > 0
    ((16, 16, 16, None, 0, 1, 1, 8, 64, -0.125, 16, 0, None), 1),
    ((16, 16, 16, None, 0, 1, 1, 8, 64, 1e-39, 16, 0, None), 1),           # 1 / sm_scale overflows
    ((16, 16, 16, None, 0, 1, 1, 8, 96, 0.125, 16, 0, None), 2),           # D not 64 / 128
    ((16, 16, 16, None, 0, 1, 1, 8, 32, 0.125, 16, 0, None), 2),
    ((None, 16, 16, None, 0, 1, 1, 8, 64, 0.125, 16, 0, None), 1),         # null q
    ((16, 16, 16, None, 0, 1, 1, 8, 64, 0.125, None, 0, None), 1),         # null out
    ((24, 16, 16, None, 0, 1, 1, 8, 64, 0.125, 16, 0, None), 1),           # q not 16-byte aligned
    ((16, 16, 16, None, 0, 1, 1, 8, 64, 0.125, 40, 0, None), 1),           # out not 16-byte aligned
    ((16, 16, 16, 18, 0, 1, 1, 8, 64, 0.125, 16, 0, None), 1),             # mask misaligned
    ((16, 16, 16, None, 0, 1, 1, 8, 64, 0.125, 16, 0, 18), 1),             # lse misaligned
    ((16, 16, 16, None, 0, 1, 1, 1 << 31, 64, 0.125, 16, 0, None), 2),     # T above 2^31 - 1
    ((16, 16, 16, None, 0, 1, 1 << 30, 1024, 64, 0.125, 16, 0, None), 2),  # 2^33 query tiles
    ((16, 16, 16, None, 0, 1 << 32, 1 << 32, 8, 64, 0.125, 16, 0, None), 2),  # B NH wraps to 0
    ((16, 16, 16, None, 0, 1 << 40, 1 << 30, 8, 64, 0.125, 16, 0, None), 2),  # B NH overflows
    ((None, None, None, None, 0, 0, 4, 8, 64, 0.125, None, 0, None), 0),   # B = 0: nothing to do
    ((None, None, None, None, 1, 2, 4, 0, 128, 0.125, None, 0, None), 0),  # T = 0: nothing to do
    ((16, 16, 16, None, 0, 1, 1, 8, 64, 0.125, 16, 7, None), 1),         # out_dtype not a ce_dtype
    ((16, 16, 16, None, 0, 1, 1, 8, 64, 0.125, 16, 1, None), 2),         # fp16 output
])
def test_attention_host_validation(cdll, args, status):
    assert cdll.ce_attention_forward(*args, None) == status


# --- the Python binding refuses caller buffers it cannot hand to a kernel -----

def test_binding_buffer_checks_on_the_host():
    # host-side checks of the binding's helpers: a buffer off the GPU, of another
    # dtype or of the wrong size is refused before any call into the library
    torch = pytest.importorskip("torch")
    from softmax_cross_entropy_online_gb300 import api
    dev = torch.device("cuda", 0)
    with pytest.raises(ValueError):
        api._check_buffer(torch.empty(3), "x", dev, torch.float32, numel=3)
    with pytest.raises(ValueError):
        api._gemm_out(torch.empty(2, 3), 2, 3, dev)
    assert api._gemm_out(None, 2, 3, torch.device("cpu")).shape == (2, 3)
    a = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        api.ce_gemm_bf16_tn(a, a)
    with pytest.raises(ValueError, match="CUDA"):
        api.ce_gemm_bf16(a, a)
    with pytest.raises(ValueError):
        api.ce_attention_forward(*(torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16),) * 3)


@pytest.mark.gpu
def test_binding_refuses_buffers_off_the_device(cdll):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_online_gb300 import api
    dev = torch.device("cuda", 0)
    n0 = api.ce_launch_count()
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError, match="out"):
        api.ce_attention_forward(q, q, q, out=torch.empty(1, 2, 8, 64))            # host
    with pytest.raises(ValueError, match="out"):
        api.ce_attention_forward(q, q, q, out=torch.empty(1, 2, 8, 32, device=dev))  # shape
    x = torch.zeros(4, 16, device=dev)
    with pytest.raises(ValueError, match="probs"):
        api.ce_softmax_forward(x, torch.empty(4, 16))
    t = torch.zeros(4, dtype=torch.int64, device=dev)
    with pytest.raises(ValueError, match="lse"):
        api.ce_backward_from_lse(x, t, torch.zeros(4), 0.25)
    with pytest.raises(ValueError, match="row_loss"):
        api.ce_fwd_bwd_inplace_noalloc(x, t, row_loss=torch.empty(4))
    a = torch.zeros(128, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError, match="D must be"):
        api.ce_gemm_bf16_tn(a, a, torch.empty(64, 128, device=dev))
    with pytest.raises(ValueError, match="D must be"):
        api.ce_gemm_bf16(a, a, torch.empty(128, 128))
    h = torch.zeros(8, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError, match="workspace"):
        api.linear_ce_fwd_bwd(h, h, torch.zeros(8, dtype=torch.int64, device=dev),
                              workspace=torch.empty(16, dtype=torch.float32, device=dev))
    torch.cuda.synchronize()
    assert api.ce_launch_count() == n0  # nothing was launched


def test_binding_rejects_an_unknown_reduction():
    torch = pytest.importorskip("torch")
    from softmax_cross_entropy_online_gb300 import api
    assert api._reduction_code("sum") == 1
    with pytest.raises(ValueError, match="reduction"):
        api._reduction_code("average")
