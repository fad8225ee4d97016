"""Python binding of the C ABI in include/ce_gb300.h (ctypes).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libce_gb300.so.  torch supplies device memory and streams.  There
is no CPU fallback: without the built library every call raises.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

from . import build as _build

CE_OK = 0
CE_ERR_INVALID_ARG = 1
CE_ERR_UNSUPPORTED = 2
CE_ERR_TARGET_RANGE = 3
CE_ERR_CUDA = 4
CE_ERR_TIMEOUT = 5

CE_F32, CE_F16, CE_BF16 = 0, 1, 2
_DTYPES = {torch.float32: CE_F32, torch.float16: CE_F16, torch.bfloat16: CE_BF16}
_DTYPE_NAMES = {"f32": CE_F32, "f16": CE_F16, "bf16": CE_BF16}
_REDUCTIONS = {"mean": 0, "sum": 1, "none": 2}

# (name, restype, argtypes) of every entry point declared in include/ce_gb300.h
_vp, _i64, _i32, _f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
SIGNATURES = {
    "ce_forward": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp]),
    "ce_fwd_bwd_inplace": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp]),
    "ce_fwd_bwd_inplace_noalloc": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp]),
    "ce_backward_from_lse": (_i32, [_vp, _vp, _vp, _i64, _i64, _i32, _f32, _vp]),
    "ce_softmax_forward": (_i32, [_vp, _vp, _i64, _i64, _i32, _vp, _vp]),
    "linear_ce_fwd_bwd": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                 ctypes.c_size_t, _vp]),
    "linear_ce_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64]),
    "linear_ce_workspace_size_fused": (ctypes.c_size_t, [_i64, _i64, _i64]),
    "ce_gemm_bf16_tn": (_i32, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _i64, _f32, _vp]),
    "ce_gemm_bf16": (_i32, [_vp, _i64, _i32, _vp, _i64, _i32, _vp, _i64, _i64, _i64, _i64, _f32,
                            _vp]),
    "ce_attention_forward": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64, _i64, _f32,
                                    _vp, _i32, _vp, _vp]),
    "ce_check_errors": (_i32, [_vp, _i32]),
    "ce_status_string": (ctypes.c_char_p, [_i32]),
    "ce_max_vocab": (_i64, [_i32]),
    "ce_launch_count": (ctypes.c_uint64, []),
    "ce_selftest_wait_timeout": (_i32, [_vp, _i32]),
}


class CEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_LIB = None


def lib() -> ctypes.CDLL:
    """Load libce_gb300.so (built in-tree by build.build()); raise if it is missing."""
    global _LIB
    if _LIB is None:
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: run softmax_cross_entropy_online_gb300.build.build() "
                "(the library has no CPU fallback)")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def status_string(status: int) -> str:
    return lib().ce_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != CE_OK:
        raise CEError(status, where)


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check_inputs(logits: torch.Tensor, targets: torch.Tensor):
    if not logits.is_cuda or logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous 2-D CUDA tensor [M, V]")
    if logits.dtype not in _DTYPES:
        raise ValueError(f"unsupported logits dtype {logits.dtype}")
    if (not targets.is_cuda or targets.dtype != torch.int64 or targets.dim() != 1
            or not targets.is_contiguous() or targets.numel() != logits.shape[0]
            or targets.device != logits.device):
        raise ValueError("targets must be a contiguous int64 CUDA tensor [M] on the logits' device")


def _reduction_code(reduction: str) -> int:
    if reduction not in _REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(_REDUCTIONS)}, not {reduction!r}")
    return _REDUCTIONS[reduction]


def _outputs(logits, reduction, row_loss, lse):
    _reduction_code(reduction)
    M = logits.shape[0]
    dev = logits.device
    loss_t = torch.empty((), dtype=torch.float32, device=dev) if reduction != "none" else None
    rl_t = torch.empty(M, dtype=torch.float32, device=dev) if row_loss else None
    lse_t = torch.empty(M, dtype=torch.float32, device=dev) if lse else None
    return loss_t, rl_t, lse_t


def _check_buffer(t, name, device, dtype, shape=None, numel=None):
    """A caller's buffer the kernels read or write: a contiguous CUDA tensor of
    `dtype` on `device` with the given shape (or element count).  Anything else
    is refused before a launch, since a kernel would write through a pointer of
    another device (or of the host) or past the end."""
    if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != device
            or t.dtype != dtype or not t.is_contiguous()
            or (shape is not None and tuple(t.shape) != tuple(shape))
            or (numel is not None and t.numel() != numel)):
        want = f"shape {tuple(shape)}" if shape is not None else f"{numel} elements"
        raise ValueError(f"{name} must be a contiguous {dtype} CUDA tensor on {device} with "
                         f"{want}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def ce_forward(logits: torch.Tensor, targets: torch.Tensor, reduction: str = "mean", *,
               row_loss: bool = True, lse: bool = True, stream=None):
    """Loss forward.  Returns (loss, row_loss, lse); unrequested entries are None."""
    _check_inputs(logits, targets)
    loss_t, rl_t, lse_t = _outputs(logits, reduction, row_loss, lse)
    M, V = logits.shape
    st = lib().ce_forward(logits.data_ptr(), targets.data_ptr(), M, V, _DTYPES[logits.dtype],
                          _reduction_code(reduction), _ptr(loss_t), _ptr(rl_t), _ptr(lse_t),
                          _stream_handle(stream, logits.device))
    _check(st, "ce_forward")
    return loss_t, rl_t, lse_t


def ce_fwd_bwd_inplace(logits: torch.Tensor, targets: torch.Tensor, reduction: str = "mean", *,
                       row_loss: bool = True, lse: bool = True, stream=None):
    """Fused forward + backward; `logits` is overwritten with the gradient."""
    _check_inputs(logits, targets)
    loss_t, rl_t, lse_t = _outputs(logits, reduction, row_loss, lse)
    M, V = logits.shape
    st = lib().ce_fwd_bwd_inplace(logits.data_ptr(), targets.data_ptr(), M, V,
                                  _DTYPES[logits.dtype], _reduction_code(reduction), _ptr(loss_t),
                                  _ptr(rl_t), _ptr(lse_t), _stream_handle(stream, logits.device))
    _check(st, "ce_fwd_bwd_inplace")
    return loss_t, rl_t, lse_t


def ce_fwd_bwd_inplace_noalloc(logits: torch.Tensor, targets: torch.Tensor,
                               reduction: str = "mean", *, loss: torch.Tensor | None = None,
                               row_loss: torch.Tensor | None = None,
                               lse: torch.Tensor | None = None, stream=None):
    """ce_fwd_bwd_inplace for callers that cannot allocate device memory: the
    library allocates nothing, and the caller passes every output buffer
    (fp32 loss [], row_loss [M], lse [M]; any may be None).  Returns them."""
    _check_inputs(logits, targets)
    M, V = logits.shape
    for t_, n, name in ((loss, 1, "loss"), (row_loss, M, "row_loss"), (lse, M, "lse")):
        if t_ is not None:
            _check_buffer(t_, name, logits.device, torch.float32, numel=n)
    st = lib().ce_fwd_bwd_inplace_noalloc(logits.data_ptr(), targets.data_ptr(), M, V,
                                          _DTYPES[logits.dtype], _reduction_code(reduction),
                                          _ptr(loss), _ptr(row_loss), _ptr(lse),
                                          _stream_handle(stream, logits.device))
    _check(st, "ce_fwd_bwd_inplace_noalloc")
    return loss, row_loss, lse


def ce_backward_from_lse(logits: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
                         scale: float, *, stream=None):
    """Gradient from a stored lse, written over `logits`."""
    _check_inputs(logits, targets)
    _check_buffer(lse, "lse", logits.device, torch.float32, numel=logits.shape[0])
    M, V = logits.shape
    st = lib().ce_backward_from_lse(logits.data_ptr(), targets.data_ptr(), lse.data_ptr(), M, V,
                                    _DTYPES[logits.dtype], float(scale),
                                    _stream_handle(stream, logits.device))
    _check(st, "ce_backward_from_lse")


def linear_ce_fwd_bwd(h: torch.Tensor, W: torch.Tensor, targets: torch.Tensor, *,
                      workspace: torch.Tensor | None = None, schedule: str = "lean",
                      stream=None):
    """Fused linear + cross-entropy: returns (loss, dH, dW) for bf16 h [M, H] and
    W [V, H]; the mean loss's gradients are fp32.  The workspace (uint8 CUDA
    tensor, whose size picks the schedule) defaults to
    linear_ce_workspace_size(M, H, V) bytes for schedule "lean" (no logits
    stored) and linear_ce_workspace_size_fused(M, H, V) for "fused"."""
    if schedule not in ("lean", "fused"):
        raise ValueError("schedule must be 'lean' or 'fused'")
    if (h.dtype != torch.bfloat16 or W.dtype != torch.bfloat16 or not h.is_cuda or not W.is_cuda
            or W.device != h.device):
        raise ValueError("h and W must be bf16 CUDA tensors on one device")
    if h.dim() != 2 or W.dim() != 2 or h.shape[1] != W.shape[1]:
        raise ValueError("h must be [M, H] and W [V, H]")
    if not h.is_contiguous() or not W.is_contiguous():
        raise ValueError("h and W must be contiguous")
    M, H = h.shape
    V = W.shape[0]
    if (targets.dtype != torch.int64 or targets.numel() != M or not targets.is_cuda
            or not targets.is_contiguous() or targets.device != h.device):
        raise ValueError("targets must be a contiguous int64 CUDA tensor [M] on h's device")
    dev = h.device
    if workspace is None:
        size = (lib().linear_ce_workspace_size(M, H, V) if schedule == "lean"
                else lib().linear_ce_workspace_size_fused(M, H, V))
        workspace = torch.empty(int(size), dtype=torch.uint8, device=dev)
    else:
        # its size in bytes is its element count: uint8 only
        _check_buffer(workspace, "workspace", dev, torch.uint8, numel=workspace.numel())
    loss = torch.empty((), dtype=torch.float32, device=dev)
    dH = torch.empty((M, H), dtype=torch.float32, device=dev)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    st = lib().linear_ce_fwd_bwd(h.data_ptr(), W.data_ptr(), targets.data_ptr(), M, H, V,
                                 loss.data_ptr(), dH.data_ptr(), dW.data_ptr(),
                                 workspace.data_ptr(), workspace.numel(),
                                 _stream_handle(stream, dev))
    _check(st, "linear_ce_fwd_bwd")
    return loss, dH, dW


def linear_ce_workspace_size(M: int, H: int, V: int) -> int:
    return int(lib().linear_ce_workspace_size(M, H, V))


def linear_ce_workspace_size_fused(M: int, H: int, V: int) -> int:
    return int(lib().linear_ce_workspace_size_fused(M, H, V))


def _check_operands(A, B):
    if not A.is_cuda or not B.is_cuda or A.device != B.device:
        raise ValueError("A and B must be CUDA tensors on one device")
    if A.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("A and B must have contiguous rows")


def _gemm_out(D, M, N, device):
    """The fp32 output [M, N] (rows contiguous, any row stride the ABI accepts)."""
    if D is None:
        return torch.empty((M, N), dtype=torch.float32, device=device)
    if (not isinstance(D, torch.Tensor) or not D.is_cuda or D.device != device
            or D.dtype != torch.float32 or D.dim() != 2 or tuple(D.shape) != (M, N)
            or D.stride(1) != 1):
        raise ValueError(f"D must be an fp32 CUDA tensor [{M}, {N}] with contiguous rows on "
                         f"{device}")
    return D


def ce_gemm_bf16_tn(A: torch.Tensor, B: torch.Tensor, D: torch.Tensor | None = None,
                    beta: float = 0.0, *, stream=None) -> torch.Tensor:
    """D = A B^T (beta 0) or D += A B^T (beta 1): A [M, K], B [N, K] bf16, D fp32."""
    if (A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16 or A.dim() != 2 or B.dim() != 2
            or A.shape[1] != B.shape[1]):
        raise ValueError("A [M, K] and B [N, K] must be bf16 with the same K")
    _check_operands(A, B)
    M, K = A.shape
    N = B.shape[0]
    D = _gemm_out(D, M, N, A.device)
    st = lib().ce_gemm_bf16_tn(A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                               D.data_ptr(), D.stride(0), M, N, K, float(beta),
                               _stream_handle(stream, A.device))
    _check(st, "ce_gemm_bf16_tn")
    return D


def ce_gemm_bf16(A: torch.Tensor, B: torch.Tensor, D: torch.Tensor | None = None,
                 beta: float = 0.0, *, a_mn: bool = False, b_mn: bool = False,
                 stream=None) -> torch.Tensor:
    """D[M, N] = sum_k A(m, k) B(n, k) (beta 0) or D += ... (beta 1), fp32.
    A is [M, K] (a_mn False) or its transpose stored [K, M] (a_mn True); B is
    [N, K] (b_mn False) or stored [K, N] (b_mn True); both bf16, rows contiguous."""
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16 or A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D bf16 tensors")
    if A.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("A and B must have contiguous rows")
    K, M = A.shape if a_mn else (A.shape[1], A.shape[0])
    Kb, N = B.shape if b_mn else (B.shape[1], B.shape[0])
    if Kb != K:
        raise ValueError("A and B must share K")
    _check_operands(A, B)
    D = _gemm_out(D, M, N, A.device)
    st = lib().ce_gemm_bf16(A.data_ptr(), A.stride(0), int(a_mn), B.data_ptr(), B.stride(0),
                            int(b_mn), D.data_ptr(), D.stride(0), M, N, K, float(beta),
                            _stream_handle(stream, A.device))
    _check(st, "ce_gemm_bf16")
    return D


def ce_attention_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         mask: torch.Tensor | None = None, *, causal: bool = False,
                         sm_scale: float | None = None, lse: bool = True, out=None,
                         out_dtype=torch.float32, stream=None):
    """Blockwise attention forward: softmax(Q K^T * sm_scale + mask [+ causal]) V.

    q, k, v: contiguous bf16 CUDA tensors [B, NH, T, D] (D 64 or 128); mask: fp32
    [T, T] or None; sm_scale defaults to 1/sqrt(D); out_dtype float32 or bfloat16
    (ignored when `out` is given).  Returns (out [B, NH, T, D], lse fp32
    [B, NH, T] or None)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if (not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous()
                or t.shape != q.shape or t.device != q.device):
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor shaped like q "
                             "[B, NH, T, D]")
    B, NH, T, D = q.shape
    if mask is not None and (mask.dtype != torch.float32 or tuple(mask.shape) != (T, T)
                             or not mask.is_contiguous() or mask.device != q.device):
        raise ValueError("mask must be a contiguous fp32 [T, T] tensor on q's device")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, NH, T, D), dtype=out_dtype, device=q.device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out must be fp32 or bf16")
    _check_buffer(out, "out", q.device, out.dtype, shape=(B, NH, T, D))
    lse_t = torch.empty((B, NH, T), dtype=torch.float32, device=q.device) if lse else None
    st = lib().ce_attention_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr(mask),
                                    int(bool(causal)), B, NH, T, D, float(sm_scale),
                                    out.data_ptr(), _DTYPES[out.dtype], _ptr(lse_t),
                                    _stream_handle(stream, q.device))
    _check(st, "ce_attention_forward")
    return out, lse_t


def ce_softmax_forward(logits: torch.Tensor, probs: torch.Tensor | None = None, *,
                       lse: bool = False, stream=None):
    """Row softmax of `logits` into `probs` (a new tensor by default; pass
    `logits` itself for in place).  Returns (probs, lse or None)."""
    if not logits.is_cuda or logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous 2-D CUDA tensor [M, V]")
    if logits.dtype not in _DTYPES:
        raise ValueError(f"unsupported logits dtype {logits.dtype}")
    if probs is None:
        probs = torch.empty_like(logits)
    _check_buffer(probs, "probs", logits.device, logits.dtype, shape=logits.shape)
    M, V = logits.shape
    lse_t = torch.empty(M, dtype=torch.float32, device=logits.device) if lse else None
    st = lib().ce_softmax_forward(logits.data_ptr(), probs.data_ptr(), M, V,
                                  _DTYPES[logits.dtype], _ptr(lse_t),
                                  _stream_handle(stream, logits.device))
    _check(st, "ce_softmax_forward")
    return probs, lse_t


def ce_check_errors(stream=None, timeout_ms: int = 10000, device=None) -> int:
    """Wait (bounded) for the stream and return the device error status (0 = CE_OK)."""
    return lib().ce_check_errors(_stream_handle(stream, device), int(timeout_ms))


def ce_max_vocab(dtype) -> int:
    code = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else _DTYPE_NAMES[dtype]
    return int(lib().ce_max_vocab(code))


def ce_launch_count() -> int:
    return int(lib().ce_launch_count())


def ce_selftest_wait_timeout(timeout_us: int, stream=None, device=None) -> int:
    return lib().ce_selftest_wait_timeout(_stream_handle(stream, device), int(timeout_us))
