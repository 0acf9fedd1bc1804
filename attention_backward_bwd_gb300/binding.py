"""ctypes binding of libattn_gb300.so (include/attn_bwd.h, include/attn_diag.h).

Argument marshalling only: torch tensors are turned into pointers and element
strides, outputs and workspace are allocated with torch (device memory), and
every step of the computation runs in the library's CUDA kernels.  There is no
CPU or PyTorch fallback: if the library is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn_gb300.so")

ATTN_FP16, ATTN_BF16 = 0, 1
STATUS = {0: "ATTN_OK", -1: "ATTN_ERR_DTYPE", -2: "ATTN_ERR_SHAPE", -3: "ATTN_ERR_STRIDE",
          -4: "ATTN_ERR_ALIGN", -5: "ATTN_ERR_NULL", -6: "ATTN_ERR_WORKSPACE",
          -7: "ATTN_ERR_CUDA", -8: "ATTN_ERR_DEVICE_TIMEOUT", -9: "ATTN_ERR_ARG"}


class AttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class AttnTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_b", ctypes.c_int64),
                ("stride_s", ctypes.c_int64), ("stride_h", ctypes.c_int64)]


class AttnOpts(ctypes.Structure):
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("softcap", ctypes.c_float), ("seqused_q", ctypes.c_void_p),
                ("seqused_k", ctypes.c_void_p)]


def _opts(window, softcap, seqused_q=None, seqused_k=None):
    """None when no option is asked for (plain entry points).  seqused_q/k:
    device int32 tensors [batch] of used lengths, or None."""
    if window is None and not softcap and seqused_q is None and seqused_k is None:
        return None
    left, right = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    return AttnOpts(left, right, float(softcap or 0.0), _ptr(seqused_q), _ptr(seqused_k))


_T = ctypes.POINTER(AttnTensor)
_P = ctypes.c_void_p
_I = ctypes.c_int
_BWD_ARGS = [_T, _T, _T, _T, _P, _T, _T, _T, _T, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I,
             _P, _P, _I, _I, _I, _P, ctypes.c_size_t, _P]

_lib = None
_lock = threading.Lock()

EXPORTS = ("attn_fwd", "attn_bwd", "attn_bwd_preprocess", "attn_bwd_main", "attn_bwd_postprocess",
           "attn_bwd_workspace_size", "attn_bwd_workspace_layout", "attn_bwd_noalloc",
           "attn_bwd_host", "attn_bwd_host_buffer_size", "attn_bwd_host_varlen",
           "attn_bwd_host_varlen_buffer_size", "attn_bwd_ex", "attn_fwd_ex",
           "attn_check_device_status",
           "attn_set_wait_timeout_ns", "attn_last_error", "attn_version", "attn_diag_mma",
           "attn_diag_wait_timeout", "attn_diag_tanh")


def lib() -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                f"g.build()'` (nvcc, sm_103a).  There is no fallback implementation.")
        L = ctypes.CDLL(LIB_PATH)
        L.attn_fwd.argtypes = [_T, _T, _T, _T, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I,
                               _P, _P, _I, _I, _P]
        L.attn_fwd.restype = _I
        L.attn_fwd_ex.argtypes = [_T, _T, _T, _T, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float,
                                  _I, _P, _P, _I, _I, ctypes.POINTER(AttnOpts), _P]
        L.attn_fwd_ex.restype = _I
        L.attn_bwd_ex.argtypes = (_BWD_ARGS[:23] + [ctypes.POINTER(AttnOpts), _I] +
                                  _BWD_ARGS[23:])
        L.attn_bwd_ex.restype = _I
        for name in ("attn_bwd", "attn_bwd_preprocess", "attn_bwd_main", "attn_bwd_postprocess"):
            f = getattr(L, name)
            f.argtypes = _BWD_ARGS
            f.restype = _I
        # attn_bwd's arguments without the workspace and its size
        L.attn_bwd_noalloc.argtypes = _BWD_ARGS[:23] + _BWD_ARGS[25:]
        L.attn_bwd_noalloc.restype = _I
        L.attn_bwd_host.argtypes = [_T, _T, _T, _T, _P, _T, _T, _T, _T, _I, _I, _I, _I, _I, _I,
                                    _I, ctypes.c_float, _I, _I, ctypes.POINTER(AttnOpts), _I, _P,
                                    ctypes.c_size_t, _P]
        L.attn_bwd_host.restype = _I
        L.attn_bwd_host_buffer_size.argtypes = [_I, _I, _I, _I, _I, _I, _I]
        L.attn_bwd_host_buffer_size.restype = ctypes.c_size_t
        L.attn_bwd_host_varlen.argtypes = [_T, _T, _T, _T, _P, _T, _T, _T, _T, _I, _I, _I, _I,
                                           _I, _I, _I, ctypes.c_float, _I, _P, _P, _I,
                                           ctypes.POINTER(AttnOpts), _I, _P, ctypes.c_size_t, _P]
        L.attn_bwd_host_varlen.restype = _I
        L.attn_bwd_host_varlen_buffer_size.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _I]
        L.attn_bwd_host_varlen_buffer_size.restype = ctypes.c_size_t
        L.attn_bwd_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I]
        L.attn_bwd_workspace_size.restype = ctypes.c_size_t
        L.attn_bwd_workspace_layout.argtypes = [_I, _I, _I, _I, _I,
                                                ctypes.POINTER(ctypes.c_size_t),
                                                ctypes.POINTER(ctypes.c_int64)]
        L.attn_bwd_workspace_layout.restype = _I
        L.attn_check_device_status.argtypes = [_P]
        L.attn_check_device_status.restype = _I
        L.attn_set_wait_timeout_ns.argtypes = [ctypes.c_int64]
        L.attn_set_wait_timeout_ns.restype = None
        L.attn_last_error.argtypes = []
        L.attn_last_error.restype = ctypes.c_char_p
        L.attn_version.argtypes = []
        L.attn_version.restype = ctypes.c_char_p
        L.attn_diag_mma.argtypes = [_I, _I, _I, _P, _P, _P, _P]
        L.attn_diag_mma.restype = _I
        L.attn_diag_tanh.argtypes = [_P, _P, _I, _P]
        L.attn_diag_tanh.restype = _I
        L.attn_diag_wait_timeout.argtypes = [ctypes.c_int64, _P]
        L.attn_diag_wait_timeout.restype = _I
        _lib = L
        return L


def _check(rc: int):
    if rc != 0:
        raise AttnError(rc, lib().attn_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return ATTN_FP16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    return 99  # rejected by the library with ATTN_ERR_DTYPE


def _desc(t: Optional[torch.Tensor]) -> AttnTensor:
    if t is None:
        return AttnTensor(None, 0, 0, 0)
    if t.dim() == 4:
        return AttnTensor(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))
    if t.dim() == 3:  # packed varlen [total, H, D]
        return AttnTensor(t.data_ptr(), 0, t.stride(0), t.stride(1))
    raise ValueError("attention tensors are [B, S, H, D] or packed [total, H, D]")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dims(q: torch.Tensor, k: torch.Tensor, cu_q, cu_k, max_q, max_k):
    if cu_q is not None:
        if q.dim() != 3 or k.dim() != 3:
            raise ValueError("varlen tensors must be packed [total, H, D]")
        batch = int(cu_q.numel()) - 1
        sq, sk = q.shape[0], k.shape[0]
        hq, d, hk = q.shape[1], q.shape[2], k.shape[1]
        if max_q is None or max_k is None:
            raise ValueError("varlen calls need max_seqlen_q and max_seqlen_k")
        return batch, sq, sk, hq, hk, d, int(max_q), int(max_k)
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("tensors must be [B, S, H, D]")
    return q.shape[0], q.shape[1], k.shape[1], q.shape[2], k.shape[2], q.shape[3], q.shape[1], k.shape[1]


def _placed(t, q, on_device: bool) -> bool:
    """On q's CUDA device (device entry points), or in host memory."""
    if on_device:
        return t.is_cuda and t.device == q.device
    return t.device.type == "cpu"


def _check_tensors(q, k, like_q, like_k, lse, ints, on_device: bool, varlen: bool):
    """Checks the library cannot make from raw pointers, made before any call:
    where each tensor lives (device memory for the device entry points, host
    memory for the host-buffer ones), that the attention tensors share q's
    dtype and have a unit stride over the head dimension, that o, dO, dQ have
    q's shape and v, dK, dV k's, that LSE is a contiguous fp32 tensor of the
    documented shape, and that the int32 arrays (cu_seqlens, seqused) are
    contiguous with an entry per sequence.  A tensor smaller than its
    arguments imply would otherwise be read or written past its end.

    ``like_q`` / ``like_k``: dicts name -> tensor or None; ``ints``: dict
    name -> (tensor or None, minimum entries)."""
    where = "CUDA tensors" if on_device else "host (CPU) tensors"
    nd = 3 if varlen else 4
    if q.dim() != nd or k.dim() != nd:
        raise AttnError(-2, f"q and k must be {'packed [total, H, D]' if varlen else '[B, S, H, D]'}"
                            f" tensors, got {tuple(q.shape)} and {tuple(k.shape)}")
    if q.shape[-1] != k.shape[-1] or (not varlen and q.shape[0] != k.shape[0]):
        raise AttnError(-2, f"q {tuple(q.shape)} and k {tuple(k.shape)} disagree on batch or D")
    named = {"q": q, "k": k, **like_q, **like_k}
    for name, t in named.items():
        if t is None:
            continue
        if not _placed(t, q, on_device):
            raise AttnError(-9, f"{name} must be {where}"
                                f"{' on ' + str(q.device) if on_device else ''}, got {t.device}")
        if t.dtype != q.dtype:
            raise AttnError(-1, f"{name} has dtype {t.dtype}, q has {q.dtype}")
        if t.numel() > 0 and t.stride(-1) != 1:
            raise AttnError(-3, f"{name} must have unit stride over the head dimension")
    for name, t in like_q.items():
        if t is not None and t.shape != q.shape:
            raise AttnError(-2, f"{name} has shape {tuple(t.shape)}, q has {tuple(q.shape)}")
    for name, t in like_k.items():
        if t is not None and t.shape != k.shape:
            raise AttnError(-2, f"{name} has shape {tuple(t.shape)}, k has {tuple(k.shape)}")
    if lse is not None:
        want = (q.shape[1], q.shape[0]) if varlen else (q.shape[0], q.shape[2], q.shape[1])
        if not _placed(lse, q, on_device):
            raise AttnError(-9, f"lse must be {where}, got {lse.device}")
        if lse.dtype != torch.float32 or tuple(lse.shape) != want or not lse.is_contiguous():
            raise AttnError(-2, f"lse must be a contiguous float32 tensor of shape {want}, got "
                                f"{lse.dtype} {tuple(lse.shape)}")
    for name, (t, n) in ints.items():
        if t is None:
            continue
        if not t.is_cuda or t.device != q.device:
            raise AttnError(-9, f"{name} must be a CUDA tensor on {q.device}, got {t.device}")
        if t.dtype != torch.int32 or not t.is_contiguous() or t.dim() != 1 or t.numel() < n:
            raise AttnError(-9, f"{name} must be a contiguous 1-D int32 tensor of at least {n} "
                                f"entries, got {t.dtype} {tuple(t.shape)}")


def version() -> str:
    return lib().attn_version().decode()


def attn_fwd(q, k, v, causal: bool = False, scale: Optional[float] = None, cu_seqlens_q=None,
             cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, out=None, lse=None,
             stream=None, window=None, softcap: float = 0.0, seqused_q=None,
             seqused_k=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Forward pass: returns (O like q, LSE fp32 [B,H,Sq] or [H,total_q], natural log).

    ``window=(left, right)`` selects a local mask (-1 = unbounded side);
    ``softcap > 0`` caps the logits as softcap * tanh(logit / softcap);
    ``seqused_q/k`` (device int32 [batch]) are per-sequence used lengths."""
    L = lib()
    b, sq, sk, hq, hk, d, mq, mk = _dims(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                                         max_seqlen_k)
    varlen = cu_seqlens_q is not None
    _check_tensors(q, k, {"out": out}, {"v": v}, lse,
                   {"cu_seqlens_q": (cu_seqlens_q, b + 1), "cu_seqlens_k": (cu_seqlens_k, b + 1),
                    "seqused_q": (seqused_q, b), "seqused_k": (seqused_k, b)}, True, varlen)
    scale = d ** -0.5 if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    if lse is None:
        shape = (hq, sq) if varlen else (b, hq, sq)
        lse = torch.empty(shape, dtype=torch.float32, device=q.device)
    dq_, dk_, dv_, do_ = _desc(q), _desc(k), _desc(v), _desc(o)
    args = [ctypes.byref(dq_), ctypes.byref(dk_), ctypes.byref(dv_), ctypes.byref(do_), _ptr(lse),
            _dtype_code(q), b, sq, sk, hq, hk, d, scale, int(bool(causal)), _ptr(cu_seqlens_q),
            _ptr(cu_seqlens_k), mq, mk]
    opts = _opts(window, softcap, seqused_q, seqused_k)
    if opts is None:
        rc = L.attn_fwd(*args, _stream(stream))
    else:
        rc = L.attn_fwd_ex(*args, ctypes.byref(opts), _stream(stream))
    _check(rc)
    return o, lse


def workspace_size(batch: int, seqlen_q: int, h_q: int, head_dim: int, deterministic: bool = False,
                   varlen: bool = False) -> int:
    return int(lib().attn_bwd_workspace_size(batch, seqlen_q, h_q, head_dim, int(deterministic),
                                             int(varlen)))


def workspace_layout(batch: int, seqlen_q: int, h_q: int, head_dim: int, varlen: bool = False):
    """Returns (offsets dict in bytes, rows)."""
    offs = (ctypes.c_size_t * 4)()
    rows = ctypes.c_int64()
    _check(lib().attn_bwd_workspace_layout(batch, seqlen_q, h_q, head_dim, int(varlen), offs,
                                           ctypes.byref(rows)))
    return {"lse2": offs[0], "delta": offs[1], "dqaccum": offs[2], "sem": offs[3]}, rows.value


def alloc_workspace(q, cu_seqlens_q=None, deterministic=False) -> torch.Tensor:
    if cu_seqlens_q is not None:
        b, sq, hq, d = int(cu_seqlens_q.numel()) - 1, q.shape[0], q.shape[1], q.shape[2]
    else:
        b, sq, hq, d = q.shape[0], q.shape[1], q.shape[2], q.shape[3]
    n = workspace_size(b, sq, hq, d, deterministic, cu_seqlens_q is not None)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


_STAGE_FN = {"all": "attn_bwd", "pre": "attn_bwd_preprocess", "main": "attn_bwd_main",
             "post": "attn_bwd_postprocess"}
_STAGE_MASK = {"all": 7, "pre": 1, "main": 2, "post": 4}


def attn_bwd(q, k, v, o, lse, do, causal: bool = False, scale: Optional[float] = None,
             cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None,
             deterministic: bool = False, workspace: Optional[torch.Tensor] = None, dq=None,
             dk=None, dv=None, stream=None, stage: str = "all", window=None,
             softcap: float = 0.0, seqused_q=None, seqused_k=None):
    """Backward pass: returns (dQ, dK, dV), each like its input.

    ``stage`` selects one of the three kernels ("pre", "main", "post") or all
    of them in order ("all"); the stages must share the workspace.
    ``window=(left, right)`` selects a local mask (-1 = unbounded side; causal
    bounds the right side at 0); ``softcap > 0`` caps the logits as
    softcap * tanh(logit / softcap) (use the forward's settings); ``seqused_q/k``
    (device int32 [batch]) are per-sequence used lengths (rows past them are
    left as they were).
    """
    L = lib()
    b, sq, sk, hq, hk, d, mq, mk = _dims(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                                         max_seqlen_k)
    _check_tensors(q, k, {"o": o, "do": do, "dq": dq}, {"v": v, "dk": dk, "dv": dv}, lse,
                   {"cu_seqlens_q": (cu_seqlens_q, b + 1), "cu_seqlens_k": (cu_seqlens_k, b + 1),
                    "seqused_q": (seqused_q, b), "seqused_k": (seqused_k, b)}, True,
                   cu_seqlens_q is not None)
    if workspace is not None and not (workspace.is_cuda and workspace.device == q.device):
        raise AttnError(-9, f"workspace must be a CUDA tensor on {q.device}")
    scale = d ** -0.5 if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = alloc_workspace(q, cu_seqlens_q, deterministic)
    descs = [_desc(t) for t in (q, k, v, o)]
    d_do, d_dq, d_dk, d_dv = _desc(do), _desc(dq), _desc(dk), _desc(dv)
    args = [*(ctypes.byref(x) for x in descs), _ptr(lse), ctypes.byref(d_do), ctypes.byref(d_dq),
            ctypes.byref(d_dk), ctypes.byref(d_dv), _dtype_code(q), b, sq, sk, hq, hk, d, scale,
            int(bool(causal)), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), mq, mk,
            int(bool(deterministic))]
    tail = [workspace.data_ptr(), workspace.numel(), _stream(stream)]
    opts = _opts(window, softcap, seqused_q, seqused_k)
    if opts is None:
        rc = getattr(L, _STAGE_FN[stage])(*args, *tail)
    else:
        rc = L.attn_bwd_ex(*args, ctypes.byref(opts), _STAGE_MASK[stage], *tail)
    _check(rc)
    return dq, dk, dv


def host_buffer_size(batch: int, seqlen_q: int, seqlen_k: int, h_q: int, h_k: int,
                     head_dim: int, chunks: int = 0) -> int:
    """Device bytes that attn_bwd_host needs for this problem and chunk count."""
    return int(lib().attn_bwd_host_buffer_size(batch, seqlen_q, seqlen_k, h_q, h_k, head_dim,
                                               chunks))


def attn_bwd_host(q, k, v, o, lse, do, dq=None, dk=None, dv=None, causal: bool = False,
                  scale: Optional[float] = None, deterministic: bool = False, chunks: int = 0,
                  device_buffer: Optional[torch.Tensor] = None, device=None, stream=None,
                  window=None, softcap: float = 0.0):
    """Backward on HOST tensors ([B, S, H, D], heads adjacent; lse [B, H_q, Sq]).

    Inputs are copied to the device, the backward runs, and dQ, dK, dV are
    copied back into host tensors (pinned, allocated here if not given), all on
    ``stream``; synchronise the stream before reading them.  ``device_buffer``
    (uint8 on the device, at least ``host_buffer_size(...)`` bytes) is
    allocated on ``device`` if not given.  Returns (dq, dk, dv).
    """
    L = lib()
    _check_tensors(q, k, {"o": o, "do": do, "dq": dq}, {"v": v, "dk": dk, "dv": dv}, lse, {},
                   False, False)
    if device_buffer is not None and not device_buffer.is_cuda:
        raise AttnError(-9, "device_buffer must be a CUDA tensor")
    b, sq, sk, hq, hk, d = q.shape[0], q.shape[1], k.shape[1], q.shape[2], k.shape[2], q.shape[3]
    scale = d ** -0.5 if scale is None else float(scale)
    pin = torch.cuda.is_available()
    dq = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin) if dq is None else dq
    dk = torch.empty(k.shape, dtype=k.dtype, pin_memory=pin) if dk is None else dk
    dv = torch.empty(v.shape, dtype=v.dtype, pin_memory=pin) if dv is None else dv
    need = host_buffer_size(b, sq, sk, hq, hk, d, chunks)
    if device_buffer is None:
        device_buffer = torch.empty(max(need, 256), dtype=torch.uint8,
                                    device=device if device is not None else "cuda")
    descs = [_desc(t) for t in (q, k, v, o)]
    d_do, d_dq, d_dk, d_dv = _desc(do), _desc(dq), _desc(dk), _desc(dv)
    opts = _opts(window, softcap)
    opts_ref = None if opts is None else ctypes.byref(opts)
    rc = L.attn_bwd_host(*(ctypes.byref(x) for x in descs), _ptr(lse), ctypes.byref(d_do),
                         ctypes.byref(d_dq), ctypes.byref(d_dk), ctypes.byref(d_dv),
                         _dtype_code(q), b, sq, sk, hq, hk, d, scale, int(bool(causal)),
                         int(bool(deterministic)), opts_ref, int(chunks), device_buffer.data_ptr(),
                         device_buffer.numel(), _stream(stream))
    _check(rc)
    return dq, dk, dv


def attn_bwd_host_varlen(q, k, v, o, lse, do, cu_seqlens_q, cu_seqlens_k, dq=None, dk=None,
                         dv=None, causal: bool = False, scale: Optional[float] = None,
                         deterministic: bool = False, chunks: int = 0,
                         device_buffer: Optional[torch.Tensor] = None, device=None, stream=None,
                         window=None, softcap: float = 0.0):
    """Backward on packed HOST tensors ([total, H, D], heads adjacent; lse
    [H_q, total_q]) with host int32 cu_seqlens; results in host tensors (pinned,
    allocated here if not given), valid once ``stream`` has passed the call."""
    L = lib()
    _check_tensors(q, k, {"o": o, "do": do, "dq": dq}, {"v": v, "dk": dk, "dv": dv}, lse, {},
                   False, True)
    if device_buffer is not None and not device_buffer.is_cuda:
        raise AttnError(-9, "device_buffer must be a CUDA tensor")
    b = int(cu_seqlens_q.numel()) - 1
    tq, tk, hq, hk, d = q.shape[0], k.shape[0], q.shape[1], k.shape[1], q.shape[2]
    scale = d ** -0.5 if scale is None else float(scale)
    cu_q = cu_seqlens_q.to(torch.int32).contiguous().cpu()
    cu_k = cu_seqlens_k.to(torch.int32).contiguous().cpu()
    pin = torch.cuda.is_available()
    dq = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin) if dq is None else dq
    dk = torch.empty(k.shape, dtype=k.dtype, pin_memory=pin) if dk is None else dk
    dv = torch.empty(v.shape, dtype=v.dtype, pin_memory=pin) if dv is None else dv
    need = int(L.attn_bwd_host_varlen_buffer_size(cu_q.data_ptr(), cu_k.data_ptr(), b, tq, tk, hq,
                                                  hk, d, chunks))
    if need == 0:
        raise AttnError(-9, L.attn_last_error().decode() or "invalid varlen arguments")
    if device_buffer is None:
        device_buffer = torch.empty(need, dtype=torch.uint8,
                                    device=device if device is not None else "cuda")
    descs = [_desc(t) for t in (q, k, v, o)]
    d_do, d_dq, d_dk, d_dv = _desc(do), _desc(dq), _desc(dk), _desc(dv)
    opts = _opts(window, softcap)
    rc = L.attn_bwd_host_varlen(*(ctypes.byref(x) for x in descs), _ptr(lse), ctypes.byref(d_do),
                                ctypes.byref(d_dq), ctypes.byref(d_dk), ctypes.byref(d_dv),
                                _dtype_code(q), b, tq, tk, hq, hk, d, scale, int(bool(causal)),
                                cu_q.data_ptr(), cu_k.data_ptr(), int(bool(deterministic)),
                                None if opts is None else ctypes.byref(opts), int(chunks),
                                device_buffer.data_ptr(), device_buffer.numel(), _stream(stream))
    _check(rc)
    return dq, dk, dv


def check_device_status(stream=None):
    """Synchronise the stream and raise if a kernel reported a device-side error."""
    _check(lib().attn_check_device_status(_stream(stream)))


def set_wait_timeout_ns(ns: int):
    lib().attn_set_wait_timeout_ns(int(ns))


def diag_mma(mode: int, a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    """Single-tile tensor-core check (see include/attn_diag.h); returns fp32 C."""
    d = b.shape[1]
    rows_c, cols_c = (128, 128) if mode == 0 else (128, d)
    c = torch.empty(rows_c, cols_c, dtype=torch.float32, device=a.device)
    _check(lib().attn_diag_mma(mode, _dtype_code(a), d, a.data_ptr(), b.data_ptr(), c.data_ptr(),
                               _stream(None)))
    return c


def diag_tanh(x: torch.Tensor) -> torch.Tensor:
    """The kernels' tanh (logit cap) on a device fp32 tensor (see include/attn_diag.h)."""
    y = torch.empty_like(x)
    _check(lib().attn_diag_tanh(x.data_ptr(), y.data_ptr(), x.numel(), _stream(None)))
    return y


def diag_wait_timeout(ns: int):
    _check(lib().attn_diag_wait_timeout(int(ns), _stream(None)))
