"""ctypes binding of liblce_gb300.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels. This module
checks dtypes/devices, allocates outputs and the workspace with PyTorch (the
library itself never allocates), passes raw pointers and the current CUDA
stream, and turns a non-zero lce_status into an exception. There is no CPU
fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build_lib import LIB_PATH

IGNORE_INDEX = -100

STATUS_NAMES = {
    0: "LCE_OK",
    1: "LCE_ERR_INVALID_ARG",
    2: "LCE_ERR_ALIGNMENT",
    3: "LCE_ERR_WORKSPACE",
    4: "LCE_ERR_LABEL_RANGE",
    5: "LCE_ERR_TIMEOUT",
    6: "LCE_ERR_CUDA",
    7: "LCE_ERR_UNSUPPORTED",
}

# Every function the C ABI (include/lce.h) exports.
EXPORTED = (
    "lce_workspace_size",
    "lce_forward",
    "lce_backward",
    "lce_fwd_bwd",
    "lce_forward_ex",
    "lce_backward_ex",
    "lce_fwd_bwd_ex",
    "lce_workspace_size_opt",
    "lce_forward_opt",
    "lce_backward_opt",
    "lce_fwd_bwd_opt",
    "lce_forward_workspace_size",
    "lce_count_valid",
    "lce_fwd_bwd_sharded",
    "lce_noalloc_read_status",
    "lce_forward_noalloc",
    "lce_ce_logits_workspace_size",
    "lce_ce_logits",
    "lce_rmsnorm_forward",
    "lce_rmsnorm_backward_workspace_size",
    "lce_rmsnorm_backward",
    "lce_norm_workspace_size",
    "lce_norm_fwd_bwd",
    "lce_norm_workspace_size_opt",
    "lce_norm_fwd_bwd_opt",
    "lce_selftest_wait_timeout",
    "lce_read_status",
    "lce_status_string",
    "lce_version",
    "lce_last_launch_count",
    "lce_profile_enable",
    "lce_profile_read",
    "lce_profile_reset",
)

KERNEL_KINDS = {"logits": 0, "grad": 1, "merge": 2, "other": 3, "norm": 4, "phase": 5, "dh": 6}
REDUCTIONS = {"mean": 0, "sum": 1, "none": 2}


class LCEError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        msg = f"{what}: {name}" if what else name
        try:
            msg += f" ({lib().lce_status_string(status).decode()})"
        except Exception:
            pass
        super().__init__(msg)


_LIB = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


def lib() -> ctypes.CDLL:
    """Load liblce_gb300.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{os.path.basename(LIB_PATH)} is not built; run "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    L = ctypes.CDLL(LIB_PATH)
    L.lce_workspace_size.argtypes = [_i64, _i64, _i64, _i64, ctypes.POINTER(ctypes.c_size_t)]
    L.lce_forward.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp,
                              ctypes.c_size_t, _vp]
    L.lce_backward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                               _vp, ctypes.c_size_t, _vp]
    L.lce_fwd_bwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp,
                              _vp, _vp, ctypes.c_size_t, _vp]
    L.lce_forward_ex.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _vp,
                                 _vp, _vp, ctypes.c_size_t, _vp]
    L.lce_backward_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                  ctypes.c_int, _vp, ctypes.c_size_t, _vp]
    L.lce_fwd_bwd_ex.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int,
                                 _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    L.lce_workspace_size_opt.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_size_t)]
    L.lce_forward_opt.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int,
                                  ctypes.c_int, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    L.lce_backward_opt.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                   ctypes.c_int, ctypes.c_int, _vp, ctypes.c_size_t, _vp]
    L.lce_fwd_bwd_opt.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int,
                                  ctypes.c_int, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    L.lce_forward_workspace_size.argtypes = [_i64, _i64, _i64, _i64,
                                             ctypes.POINTER(ctypes.c_size_t)]
    L.lce_count_valid.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp]
    L.lce_fwd_bwd_sharded.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                      ctypes.c_int, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    L.lce_noalloc_read_status.argtypes = [_vp]
    L.lce_forward_noalloc.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp]
    L.lce_ce_logits_workspace_size.argtypes = [_i64, ctypes.POINTER(ctypes.c_size_t)]
    L.lce_ce_logits.argtypes = [_vp, ctypes.c_int, _i64, _vp, _i64, _i64, _i64, ctypes.c_int, _vp,
                                _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    _f = ctypes.c_float
    _sz = ctypes.POINTER(ctypes.c_size_t)
    L.lce_rmsnorm_forward.argtypes = [_vp, _vp, _i64, _i64, _f, _vp, _vp, _vp]
    L.lce_rmsnorm_backward_workspace_size.argtypes = [_i64, _sz]
    L.lce_rmsnorm_backward.argtypes = [_vp, _vp, _vp, ctypes.c_int, _i64, _i64, _f, _vp, _vp, _vp,
                                       ctypes.c_size_t, _vp]
    L.lce_norm_workspace_size.argtypes = [_i64, _i64, _i64, _i64, _sz]
    L.lce_norm_fwd_bwd.argtypes = [_vp, _vp, _f, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                   ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    L.lce_norm_workspace_size_opt.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int, _sz]
    L.lce_norm_fwd_bwd_opt.argtypes = [_vp, _vp, _f, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                       ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp,
                                       ctypes.c_size_t, _vp]
    L.lce_selftest_wait_timeout.argtypes = [_vp, ctypes.c_size_t, _i64, _vp]
    L.lce_read_status.argtypes = [_vp, _vp]
    L.lce_status_string.argtypes = [ctypes.c_int]
    L.lce_status_string.restype = ctypes.c_char_p
    L.lce_version.argtypes = []
    L.lce_last_launch_count.argtypes = []
    L.lce_profile_enable.argtypes = [ctypes.c_int]
    L.lce_profile_read.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_int64)]
    L.lce_profile_reset.argtypes = []
    L.lce_profile_reset.restype = None
    for name in ("lce_profile_enable", "lce_profile_read", "lce_workspace_size", "lce_forward",
                 "lce_backward", "lce_fwd_bwd", "lce_forward_ex", "lce_backward_ex",
                 "lce_fwd_bwd_ex", "lce_read_status", "lce_version", "lce_last_launch_count",
                 "lce_ce_logits_workspace_size", "lce_ce_logits", "lce_rmsnorm_forward",
                 "lce_workspace_size_opt", "lce_forward_opt", "lce_backward_opt", "lce_fwd_bwd_opt",
                 "lce_selftest_wait_timeout",
                 "lce_rmsnorm_backward_workspace_size", "lce_rmsnorm_backward",
                 "lce_norm_workspace_size", "lce_norm_fwd_bwd", "lce_norm_workspace_size_opt",
                 "lce_norm_fwd_bwd_opt", "lce_forward_workspace_size", "lce_count_valid",
                 "lce_fwd_bwd_sharded", "lce_noalloc_read_status", "lce_forward_noalloc"):
        getattr(L, name).restype = ctypes.c_int
    _LIB = L
    return L


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st: int, what: str):
    if st != 0:
        raise LCEError(st, what)


def workspace_size(N: int, D: int, V: int, chunk: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().lce_workspace_size(N, D, V, chunk, ctypes.byref(out)), "lce_workspace_size")
    return out.value


ACCUMULATE = {"dW": 1, "dH": 2}
INPUT_FP16 = 4
FROZEN_W = 8
LOW_MEMORY = 16


def _acc_flags(accumulate, dH, dW, compute_dW=True) -> int:
    flags = 0
    for name in accumulate:
        if name not in ACCUMULATE:
            raise ValueError(f"accumulate takes a subset of {sorted(ACCUMULATE)}, not {name!r}")
        flags |= ACCUMULATE[name]
    if (flags & 1 and dW is None) or (flags & 2 and dH is None):
        raise ValueError("accumulating needs the existing dW / dH tensors passed in")
    if not compute_dW:
        if flags & 1:
            raise ValueError("compute_dW=False (frozen W) cannot accumulate into dW")
        flags |= FROZEN_W
    return flags


def forward_workspace_size(N: int, D: int, V: int, chunk: int) -> int:
    """Workspace bytes of lce_forward (no chunk buffer)."""
    out = ctypes.c_size_t(0)
    _check(lib().lce_forward_workspace_size(N, D, V, chunk, ctypes.byref(out)),
           "lce_forward_workspace_size")
    return out.value


def workspace_size_opt(N: int, D: int, V: int, chunk: int, flags: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().lce_workspace_size_opt(N, D, V, chunk, flags, ctypes.byref(out)),
           "lce_workspace_size_opt")
    return out.value


def alloc_workspace(N: int, D: int, V: int, chunk: int, device, flags: int = 0) -> torch.Tensor:
    return torch.empty(workspace_size_opt(N, D, V, chunk, flags), dtype=torch.uint8, device=device)


def _check_inputs(H, W, y):
    if not (H.is_cuda and W.is_cuda and y.is_cuda):
        raise ValueError("H, W and y must be CUDA tensors (there is no CPU path)")
    if H.dtype not in (torch.bfloat16, torch.float16) or W.dtype != H.dtype:
        raise TypeError("H and W must both be bfloat16 or both float16")
    if y.dtype != torch.int64:
        raise TypeError("y must be int64")
    if H.dim() != 2 or W.dim() != 2 or y.dim() != 1:
        raise ValueError("expected H[N,D], W[V,D], y[N]")
    if H.shape[1] != W.shape[1] or H.shape[0] != y.shape[0]:
        raise ValueError(f"shape mismatch: H{tuple(H.shape)} W{tuple(W.shape)} y{tuple(y.shape)}")
    if not (H.is_contiguous() and W.is_contiguous() and y.is_contiguous()):
        raise ValueError("H, W and y must be contiguous")
    return H.shape[0], H.shape[1], W.shape[0]


def _reduction(reduction: str) -> int:
    if reduction not in REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(REDUCTIONS)}")
    return REDUCTIONS[reduction]


def _loss_buffer(loss, N, reduction, dev):
    if loss is None:
        loss = torch.empty(N if reduction == "none" else 1, dtype=torch.float32, device=dev)
    return loss


def _check_dloss(dloss, N, reduction):
    if dloss is None:
        return
    if dloss.dtype != torch.float32 or not dloss.is_cuda or not dloss.is_contiguous():
        raise TypeError("dloss must be a contiguous CUDA float32 tensor")
    want = N if reduction == "none" else 1
    if dloss.numel() != want:
        raise ValueError(f"dloss must have {want} element(s) for reduction={reduction!r}")


def lce_forward(H, W, y, chunk: int = 1024, ignore_index: int = IGNORE_INDEX,
                loss=None, lse=None, ws=None, stream=None, reduction: str = "mean"):
    """Loss (device scalar, or [N] for reduction="none") and lse[N]."""
    N, D, V = _check_inputs(H, W, y)
    dev = H.device
    red = _reduction(reduction)
    loss = _loss_buffer(loss, N, reduction, dev)
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    if ws is None:
        ws = torch.empty(forward_workspace_size(N, D, V, chunk), dtype=torch.uint8, device=dev)
    flags = INPUT_FP16 if H.dtype == torch.float16 else 0
    st = lib().lce_forward_opt(_ptr(H), _ptr(W), _ptr(y), N, D, V, ignore_index, chunk, red, flags,
                               _ptr(loss), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "lce_forward")
    return loss, lse


def lce_backward(H, W, y, lse, dloss=None, chunk: int = 1024, ignore_index: int = IGNORE_INDEX,
                 dH=None, dW=None, ws=None, stream=None, reduction: str = "mean",
                 accumulate=(), compute_dW: bool = True, low_memory: bool = False):
    """dH (bf16) and dW (fp32) from a saved lse. dloss: scalar tensor, or [N] for
    reduction="none"; None means 1. accumulate: a subset of ("dW", "dH") added
    into the given dW / dH instead of overwriting them. compute_dW=False: W is
    frozen, dW is neither computed nor returned (None). low_memory: one chunk
    buffer (LCE_LOW_MEMORY: one dW contraction per chunk)."""
    N, D, V = _check_inputs(H, W, y)
    dev = H.device
    red = _reduction(reduction)
    flags = (_acc_flags(accumulate, dH, dW, compute_dW) |
             (INPUT_FP16 if H.dtype == torch.float16 else 0) | (LOW_MEMORY if low_memory else 0))
    if dH is None:
        dH = torch.empty(N, D, dtype=H.dtype, device=dev)
    if not compute_dW:
        dW = None
    elif dW is None:
        dW = torch.empty(V, D, dtype=torch.float32, device=dev)
    if ws is None:
        ws = alloc_workspace(N, D, V, chunk, dev, flags)
    _check_dloss(dloss, N, reduction)
    st = lib().lce_backward_opt(_ptr(H), _ptr(W), _ptr(y), _ptr(lse), _ptr(dloss), _ptr(dH),
                                _ptr(dW), N, D, V, ignore_index, chunk, red, flags, _ptr(ws),
                                ws.numel(), _stream(stream))
    _check(st, "lce_backward")
    return dH, dW


def lce_fwd_bwd(H, W, y, dloss=None, chunk: int = 1024, ignore_index: int = IGNORE_INDEX,
                loss=None, lse=None, dH=None, dW=None, ws=None, stream=None,
                reduction: str = "mean", accumulate=(), compute_dW: bool = True,
                n_valid_total=None, low_memory: bool = False):
    """Fused forward + backward: (loss, lse, dH, dW). accumulate: a subset of
    ("dW", "dH") added into the given dW / dH instead of overwriting them.
    compute_dW=False: W is frozen (e.g. a LoRA fine-tune), dW is None.
    n_valid_total: a device int64 tensor of one element, the valid rows of every
    shard of a token-sharded batch (reduction "mean" only): the mean divides by
    it instead of this call's count (lce_fwd_bwd_sharded). low_memory: one chunk
    buffer (LCE_LOW_MEMORY: about half the workspace, one dW contraction per chunk
    instead of one per pair of chunks)."""
    N, D, V = _check_inputs(H, W, y)
    dev = H.device
    red = _reduction(reduction)
    flags = (_acc_flags(accumulate, dH, dW, compute_dW) |
             (INPUT_FP16 if H.dtype == torch.float16 else 0) | (LOW_MEMORY if low_memory else 0))
    loss = _loss_buffer(loss, N, reduction, dev)
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    if dH is None:
        dH = torch.empty(N, D, dtype=H.dtype, device=dev)
    if not compute_dW:
        dW = None
    elif dW is None:
        dW = torch.empty(V, D, dtype=torch.float32, device=dev)
    if ws is None:
        ws = alloc_workspace(N, D, V, chunk, dev, flags)
    _check_dloss(dloss, N, reduction)
    if n_valid_total is not None:
        if reduction != "mean":
            raise ValueError("n_valid_total is the normaliser of the mean: reduction must be 'mean'")
        if (n_valid_total.dtype != torch.int64 or not n_valid_total.is_cuda
                or n_valid_total.numel() != 1):
            raise TypeError("n_valid_total must be a CUDA int64 tensor of one element")
        st = lib().lce_fwd_bwd_sharded(_ptr(H), _ptr(W), _ptr(y), _ptr(dloss), _ptr(n_valid_total),
                                       N, D, V, ignore_index, chunk, flags, _ptr(loss), _ptr(lse),
                                       _ptr(dH), _ptr(dW), _ptr(ws), ws.numel(), _stream(stream))
        _check(st, "lce_fwd_bwd_sharded")
        return loss, lse, dH, dW
    st = lib().lce_fwd_bwd_opt(_ptr(H), _ptr(W), _ptr(y), _ptr(dloss), N, D, V, ignore_index,
                               chunk, red, flags, _ptr(loss), _ptr(lse), _ptr(dH), _ptr(dW),
                               _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "lce_fwd_bwd")
    return loss, lse, dH, dW


def count_valid(y, V: int, ignore_index: int = IGNORE_INDEX, out=None, stream=None):
    """Rows of y whose label lies in [0, V) and is not ignore_index, counted on the
    device by the library (lce_count_valid): an int64 CUDA tensor of one element."""
    if not y.is_cuda:
        raise ValueError("y must be a CUDA tensor (there is no CPU path)")
    if y.dtype != torch.int64 or y.dim() != 1 or not y.is_contiguous():
        raise TypeError("y must be a contiguous int64 vector")
    if out is None:
        out = torch.empty(1, dtype=torch.int64, device=y.device)
    _check(lib().lce_count_valid(_ptr(y), y.shape[0], V, ignore_index, _ptr(out), _stream(stream)),
           "lce_count_valid")
    return out


_CE_DTYPES = {torch.bfloat16: 0, torch.float32: 1, torch.float16: 2}


def ce_logits(Z, y, dloss=None, ignore_index: int = IGNORE_INDEX, reduction: str = "mean",
              grad: bool = True, inplace: bool = False, loss=None, lse=None, ws=None, stream=None):
    """Cross-entropy over precomputed logits Z [N, V] (bf16, fp16 or fp32, row stride may
    exceed V): (loss, lse, dZ). dZ is None when grad is False; with inplace=True
    it overwrites Z."""
    if not (Z.is_cuda and y.is_cuda):
        raise ValueError("Z and y must be CUDA tensors (there is no CPU path)")
    if Z.dtype not in _CE_DTYPES or y.dtype != torch.int64:
        raise TypeError("Z must be bfloat16, float16 or float32 and y int64")
    if Z.dim() != 2 or Z.stride(1) != 1 or y.dim() != 1 or y.shape[0] != Z.shape[0]:
        raise ValueError("expected Z[N, V] with unit column stride and y[N]")
    N, V = Z.shape
    ld = Z.stride(0) if N > 1 else V
    dev = Z.device
    red = _reduction(reduction)
    loss = _loss_buffer(loss, N, reduction, dev)
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    dZ = None
    if grad:
        dZ = Z if inplace else torch.empty_strided(Z.shape, Z.stride(), dtype=Z.dtype, device=dev)
    if ws is None:
        nbytes = ctypes.c_size_t(0)
        _check(lib().lce_ce_logits_workspace_size(N, ctypes.byref(nbytes)), "workspace")
        ws = torch.empty(nbytes.value, dtype=torch.uint8, device=dev)
    _check_dloss(dloss, N, reduction)
    st = lib().lce_ce_logits(_ptr(Z), _CE_DTYPES[Z.dtype], ld, _ptr(y), N, V,
                             ignore_index, red, _ptr(dloss), _ptr(loss), _ptr(lse), _ptr(dZ),
                             _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "lce_ce_logits")
    return loss, lse, dZ


def _check_norm_inputs(X, gamma):
    if not (X.is_cuda and gamma.is_cuda):
        raise ValueError("X and gamma must be CUDA tensors (there is no CPU path)")
    if X.dtype != torch.bfloat16 or gamma.dtype != torch.bfloat16:
        raise TypeError("X and gamma must be bfloat16")
    if X.dim() != 2 or gamma.dim() != 1 or gamma.shape[0] != X.shape[1]:
        raise ValueError("expected X[N, D] and gamma[D]")
    if not (X.is_contiguous() and gamma.is_contiguous()):
        raise ValueError("X and gamma must be contiguous")


def rmsnorm_forward(X, gamma, eps: float = 1e-6, want_rstd: bool = False, stream=None):
    """H = X / sqrt(mean(X^2) + eps) * gamma (bf16); with want_rstd also r [N] fp32."""
    _check_norm_inputs(X, gamma)
    N, D = X.shape
    H = torch.empty_like(X)
    rstd = torch.empty(N, dtype=torch.float32, device=X.device) if want_rstd else None
    _check(lib().lce_rmsnorm_forward(_ptr(X), _ptr(gamma), N, D, eps, _ptr(H), _ptr(rstd),
                                     _stream(stream)), "lce_rmsnorm_forward")
    return (H, rstd) if want_rstd else H


def rmsnorm_backward(X, gamma, dH, eps: float = 1e-6, ws=None, stream=None):
    """(dX bf16, dgamma fp32) of RMSNorm for the upstream gradient dH (bf16 or fp32)."""
    _check_norm_inputs(X, gamma)
    if dH.shape != X.shape or dH.dtype not in (torch.bfloat16, torch.float32) or not dH.is_contiguous():
        raise ValueError("dH must be a contiguous bf16 or fp32 tensor shaped like X")
    N, D = X.shape
    dX = torch.empty_like(X)
    dgamma = torch.empty(D, dtype=torch.float32, device=X.device)
    if ws is None:
        nbytes = ctypes.c_size_t(0)
        _check(lib().lce_rmsnorm_backward_workspace_size(D, ctypes.byref(nbytes)), "workspace")
        ws = torch.empty(nbytes.value, dtype=torch.uint8, device=X.device)
    _check(lib().lce_rmsnorm_backward(_ptr(X), _ptr(gamma), _ptr(dH),
                                      1 if dH.dtype == torch.float32 else 0, N, D, eps, _ptr(dX),
                                      _ptr(dgamma), _ptr(ws), ws.numel(), _stream(stream)),
           "lce_rmsnorm_backward")
    return dX, dgamma


def norm_workspace_size(N: int, D: int, V: int, chunk: int, flags: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().lce_norm_workspace_size_opt(N, D, V, chunk, flags, ctypes.byref(out)),
           "lce_norm_workspace_size_opt")
    return out.value


def norm_fwd_bwd(X, gamma, W, y, eps: float = 1e-6, dloss=None, chunk: int = 1024,
                 ignore_index: int = IGNORE_INDEX, reduction: str = "mean", ws=None, loss=None,
                 lse=None, stream=None, compute_dW: bool = True, low_memory: bool = False):
    """RMSNorm + LM head + cross-entropy, forward and backward in one call:
    (loss, lse, dX bf16, dgamma fp32, dW fp32). compute_dW=False: W is frozen and
    dW is None. low_memory: one chunk buffer (LCE_LOW_MEMORY)."""
    _check_norm_inputs(X, gamma)
    _check_inputs(X, W, y)
    N, D = X.shape
    V = W.shape[0]
    dev = X.device
    red = _reduction(reduction)
    loss = _loss_buffer(loss, N, reduction, dev)
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    dX = torch.empty_like(X)
    dgamma = torch.empty(D, dtype=torch.float32, device=dev)
    flags = (0 if compute_dW else FROZEN_W) | (LOW_MEMORY if low_memory else 0)
    dW = torch.empty(V, D, dtype=torch.float32, device=dev) if compute_dW else None
    if ws is None:
        ws = torch.empty(norm_workspace_size(N, D, V, chunk, flags), dtype=torch.uint8, device=dev)
    _check_dloss(dloss, N, reduction)
    _check(lib().lce_norm_fwd_bwd_opt(_ptr(X), _ptr(gamma), eps, _ptr(W), _ptr(y), _ptr(dloss), N,
                                      D, V, ignore_index, chunk, red, flags, _ptr(loss), _ptr(lse),
                                      _ptr(dX), _ptr(dgamma), _ptr(dW), _ptr(ws), ws.numel(),
                                      _stream(stream)),
           "lce_norm_fwd_bwd_opt")
    return loss, lse, dX, dgamma, dW


class NormLinearCrossEntropyFunction(torch.autograd.Function):
    """loss = CE(RMSNorm(X; gamma) W^T, y) with reduction mean or sum. The forward
    runs lce_norm_fwd_bwd (gradients for an upstream gradient of 1); the backward
    scales them by the incoming gradient, which the loss is linear in. A W
    without requires_grad is frozen (no dW work)."""

    @staticmethod
    def forward(ctx, X, gamma, W, y, eps, chunk, ignore_index, reduction):
        need_dW = ctx.needs_input_grad[2]
        loss, _, dX, dgamma, dW = norm_fwd_bwd(X, gamma, W, y, eps=eps, chunk=chunk,
                                               ignore_index=ignore_index, reduction=reduction,
                                               compute_dW=need_dW)
        ctx.save_for_backward(dX, dgamma, dW)
        ctx.dtypes = (gamma.dtype, W.dtype)
        return loss.reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        dX, dgamma, dW = ctx.saved_tensors
        g = grad_out.to(torch.float32)
        return ((dX.float() * g).to(dX.dtype), (dgamma * g).to(ctx.dtypes[0]),
                (dW * g).to(ctx.dtypes[1]) if dW is not None else None,
                None, None, None, None, None)


def norm_linear_cross_entropy(X, gamma, W, y, eps: float = 1e-6, chunk: int = 1024,
                              ignore_index: int = IGNORE_INDEX, reduction: str = "mean"):
    """Differentiable CE(RMSNorm(X) W^T, y) for reduction mean / sum (the per-row
    reduction needs the upstream gradient before the backward: call norm_fwd_bwd)."""
    if reduction not in ("mean", "sum"):
        raise ValueError("norm_linear_cross_entropy supports reduction 'mean' or 'sum'")
    return NormLinearCrossEntropyFunction.apply(X, gamma, W, y, eps, chunk, ignore_index, reduction)


def selftest_wait_timeout(ws: torch.Tensor, limit_us: int = 20000, stream=None):
    """Runs the bounded-wait self-test kernel (a wait nothing ends) on ws's device."""
    _check(lib().lce_selftest_wait_timeout(_ptr(ws), ws.numel(), limit_us, _stream(stream)),
           "lce_selftest_wait_timeout")


def read_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device-side status."""
    return lib().lce_read_status(_ptr(ws), _stream(stream))


def forward_noalloc(H, W, y, loss, lse, chunk: int = 1024, ignore_index: int = IGNORE_INDEX,
                    stream=None):
    """lce_forward on the library's built-in scratch array (lce_forward_noalloc):
    the caller passes the outputs (loss [1] and lse [N], fp32) and no workspace;
    nothing is allocated, by the library or here."""
    N, D, V = _check_inputs(H, W, y)
    _check(lib().lce_forward_noalloc(_ptr(H), _ptr(W), _ptr(y), N, D, V, ignore_index, chunk,
                                     _ptr(loss), _ptr(lse), _stream(stream)),
           "lce_forward_noalloc")
    return loss, lse


def noalloc_read_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device-side status of the
    built-in scratch array used by forward_noalloc."""
    return lib().lce_noalloc_read_status(_stream(stream))


def last_launch_count() -> int:
    return lib().lce_last_launch_count()


def profile_enable(on: bool = True):
    _check(lib().lce_profile_enable(1 if on else 0), "lce_profile_enable")


def profile_reset():
    lib().lce_profile_reset()


def profile_read(kind: str):
    """(total_ms, launches) of every completed launch of one kernel kind."""
    ms = ctypes.c_double(0)
    n = ctypes.c_int64(0)
    _check(lib().lce_profile_read(KERNEL_KINDS[kind], ctypes.byref(ms), ctypes.byref(n)),
           "lce_profile_read")
    return ms.value, n.value


class LinearCrossEntropyFunction(torch.autograd.Function):
    """autograd wrapper, two schedules.

    fused (reduction mean or sum, the default): the forward runs lce_fwd_bwd for an
    upstream gradient of 1 and keeps dH and dW; the backward scales them by the
    incoming gradient, which the loss is linear in. 6NDV flops per step. The LM
    head's loss is the first node its backward reaches, so the gradients are
    held only until then.

    recompute (reduction none, whose per-row incoming gradient is unknown in the
    forward, or fused=False): forward = lce_forward keeping lse, backward =
    lce_backward recomputing the logits. 8NDV flops.

    A W that does not require grad is frozen: no dW is computed (LCE_FROZEN_W)."""

    @staticmethod
    def forward(ctx, H, W, y, chunk=1024, ignore_index=IGNORE_INDEX, reduction="mean",
                fused=True):
        need_dH, need_dW = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        ctx.fused = bool(fused) and reduction != "none" and (need_dH or need_dW)
        ctx.need_dW = need_dW
        ctx.w_dtype = W.dtype
        if ctx.fused:
            loss, _, dH, dW = lce_fwd_bwd(H, W, y, chunk=chunk, ignore_index=ignore_index,
                                          reduction=reduction, compute_dW=need_dW)
            ctx.save_for_backward(dH, dW)
        else:
            loss, lse = lce_forward(H, W, y, chunk=chunk, ignore_index=ignore_index,
                                    reduction=reduction)
            ctx.save_for_backward(H, W, y, lse)
        ctx.chunk = chunk
        ctx.ignore_index = ignore_index
        ctx.reduction = reduction
        return loss if reduction == "none" else loss.view(())

    @staticmethod
    def backward(ctx, grad_out):
        if ctx.fused:
            dH, dW = ctx.saved_tensors
            g = grad_out.detach().to(torch.float32)
            gH = (dH.float() * g).to(dH.dtype) if ctx.needs_input_grad[0] else None
            gW = (dW * g).to(ctx.w_dtype) if dW is not None else None
            return gH, gW, None, None, None, None, None
        H, W, y, lse = ctx.saved_tensors
        g = grad_out.detach().reshape(-1).to(torch.float32).contiguous()
        dH, dW = lce_backward(H, W, y, lse, dloss=g, chunk=ctx.chunk,
                              ignore_index=ctx.ignore_index, reduction=ctx.reduction,
                              compute_dW=ctx.need_dW)
        return dH, (dW.to(W.dtype) if dW is not None else None), None, None, None, None, None


def linear_cross_entropy(H, W, y, chunk: int = 1024, ignore_index: int = IGNORE_INDEX,
                         reduction: str = "mean", fused: bool = True):
    """Cross-entropy of softmax(H W^T) against y (mean, sum or per-row), differentiable
    in H and W (a W with requires_grad False is treated as frozen: no dW work).
    fused: compute the gradients in the forward pass (reductions mean and sum)."""
    return LinearCrossEntropyFunction.apply(H, W, y, chunk, ignore_index, reduction, fused)
