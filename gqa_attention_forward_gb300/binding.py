"""ctypes binding of libgqa_attn.so (argument marshalling only).

Every step of the attention forward runs inside the library's CUDA kernel;
this module converts Python / torch arguments to the C ABI declared in
``include/gqa_attn.h`` and turns status codes into exceptions.  There is no
fallback: if the library is missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import build as _build

ATTN_F16, ATTN_BF16 = 0, 1
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_NULL", 2: "ATTN_ERR_SHAPE", 3: "ATTN_ERR_HEADDIM",
          4: "ATTN_ERR_DTYPE", 5: "ATTN_ERR_ALIGN", 6: "ATTN_ERR_LAUNCH", 7: "ATTN_ERR_TIMEOUT",
          8: "ATTN_ERR_NODEVICE", 9: "ATTN_ERR_SCRATCH"}
ATTN_OK, ATTN_ERR_TIMEOUT, ATTN_ERR_SCRATCH = 0, 7, 9

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def load(path: str | None = None):
    """Load the built library (no build here: a missing library is an error)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is not built; call gqa_attention_forward_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i = ctypes.c_void_p, ctypes.c_int
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, i, vp]
        lib.attn_fwd.restype = i
        lib.attn_fwd_kv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, i, i, vp]
        lib.attn_fwd_kv.restype = i
        lib.attn_fwd_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, i, i,
                                        vp, ctypes.c_size_t, vp]
        lib.attn_fwd_decode.restype = i
        lib.attn_fwd_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float,
                                                i, i, vp]
        lib.attn_fwd_decode_noalloc.restype = i
        lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                      ctypes.c_float, i, i, vp]
        lib.attn_fwd_host.restype = i
        lib.attn_fwd_decode_workspace.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        lib.attn_fwd_decode_workspace.restype = i
        lib.attn_fwd_kv_split.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, i, i,
                                          vp, ctypes.c_size_t, vp]
        lib.attn_fwd_kv_split.restype = i
        lib.attn_fwd_kv_split_workspace.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        lib.attn_fwd_kv_split_workspace.restype = i
        lib.attn_test_force_splits.argtypes = [i]
        lib.attn_test_force_splits.restype = None
        lib.attn_status_str.argtypes = [i]
        lib.attn_status_str.restype = ctypes.c_char_p
        lib.attn_last_device_error.argtypes = [vp]
        lib.attn_last_device_error.restype = i
        lib.attn_last_cuda_error.argtypes = []
        lib.attn_last_cuda_error.restype = ctypes.c_char_p
        lib.attn_version.argtypes = []
        lib.attn_version.restype = i
        lib.attn_test_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
        lib.attn_test_set_wait_timeout_ns.restype = None
        lib.attn_test_inject_stall.argtypes = [i]
        lib.attn_test_inject_stall.restype = None
        lib.attn_test_select_kernel.argtypes = [i]
        lib.attn_test_select_kernel.restype = None
        lib.attn_test_set_item_order.argtypes = [i]
        lib.attn_test_set_item_order.restype = None
        if path is None:
            _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    name = str(dtype)
    if name in ("f16", "torch.float16", "float16"):
        return ATTN_F16
    if name in ("bf16", "torch.bfloat16", "bfloat16"):
        return ATTN_BF16
    return -1


def _stream_handle(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, D, scale, causal, dtype, stream=None) -> int:
    """The C entry point with the same name; returns its status code."""
    lib = load()
    return lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv),
                        int(N), int(D), float(scale), int(bool(causal)), _dtype_code(dtype),
                        _stream_handle(stream))


def attn_fwd_kv(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype, stream=None) -> int:
    """The C entry point with the same name; returns its status code."""
    lib = load()
    return lib.attn_fwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                           int(Hkv), int(Nq), int(Nk), int(D), float(scale), int(bool(causal)),
                           _dtype_code(dtype), _stream_handle(stream))


def attn_fwd_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype, workspace,
                    workspace_bytes, stream=None) -> int:
    """The C entry point with the same name; returns its status code."""
    lib = load()
    return lib.attn_fwd_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                               int(Hkv), int(Nq), int(Nk), int(D), float(scale), int(bool(causal)),
                               _dtype_code(dtype), _ptr(workspace), int(workspace_bytes),
                               _stream_handle(stream))


def attn_fwd_kv_split(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype, workspace,
                      workspace_bytes, stream=None) -> int:
    """The C entry point with the same name; returns its status code."""
    lib = load()
    return lib.attn_fwd_kv_split(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                                 int(Hkv), int(Nq), int(Nk), int(D), float(scale), int(bool(causal)),
                                 _dtype_code(dtype), _ptr(workspace), int(workspace_bytes),
                                 _stream_handle(stream))


def attn_fwd_kv_split_workspace(B, Hq, Hkv, Nq, Nk, D, causal):
    """(status, bytes) of the C entry point with the same name."""
    n = ctypes.c_size_t(0)
    st = load().attn_fwd_kv_split_workspace(int(B), int(Hq), int(Hkv), int(Nq), int(Nk), int(D),
                                            int(bool(causal)), ctypes.byref(n))
    return st, n.value


def attn_fwd_decode_noalloc(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype,
                            stream=None) -> int:
    """The C entry point with the same name; returns its status code."""
    lib = load()
    return lib.attn_fwd_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                       int(Hq), int(Hkv), int(Nq), int(Nk), int(D), float(scale),
                                       int(bool(causal)), _dtype_code(dtype), _stream_handle(stream))


def attn_fwd_host(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d, B, Hq, Hkv, Nq, Nk, D,
                  scale, causal, dtype, stream=None) -> int:
    """The C entry point with the same name; returns its status code.  Host
    arguments are CPU tensors (pinned for overlap), device arguments CUDA tensors."""
    lib = load()
    return lib.attn_fwd_host(_ptr(q_h), _ptr(k_h), _ptr(v_h), _ptr(o_h), _ptr(lse_h), _ptr(q_d),
                             _ptr(k_d), _ptr(v_d), _ptr(o_d), _ptr(lse_d), int(B), int(Hq), int(Hkv),
                             int(Nq), int(Nk), int(D), float(scale), int(bool(causal)),
                             _dtype_code(dtype), _stream_handle(stream))


def attn_fwd_decode_workspace(B, Hq, Hkv, Nq, Nk, D):
    """(status, bytes) of the C entry point with the same name."""
    n = ctypes.c_size_t(0)
    st = load().attn_fwd_decode_workspace(int(B), int(Hq), int(Hkv), int(Nq), int(Nk), int(D),
                                          ctypes.byref(n))
    return st, n.value


def attention_decode(q, k, v, causal: bool = True, scale: float | None = None,
                     with_lse: bool = True, workspace=None, out=None, lse_out=None, stream=None):
    """attn_fwd_decode for torch CUDA tensors q [B,Hq,Nq,D], k/v [B,Hkv,Nk,D].

    ``workspace``: a uint8 CUDA tensor, or None to let torch allocate the size
    attn_fwd_decode_workspace asks for.  Returns (o, lse) without waiting."""
    import torch

    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous [B, H, N, D]")
    o = out if out is not None else torch.empty_like(q)
    lse = None
    if with_lse:
        lse = lse_out if lse_out is not None else torch.empty((B, Hq, Nq), dtype=torch.float32,
                                                              device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if workspace is None:
        st, nbytes = attn_fwd_decode_workspace(B, Hq, Hkv, Nq, Nk, D)
        if st != ATTN_OK:
            raise AttnError(st, "attn_fwd_decode_workspace")
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = attn_fwd_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, q.dtype,
                         workspace, workspace.numel(), stream)
    if st != ATTN_OK:
        raise AttnError(st, f"attn_fwd_decode ({attn_last_cuda_error()})")
    return o, lse


def attention_split(q, k, v, causal: bool = True, scale: float | None = None, with_lse: bool = True,
                    workspace=None, out=None, lse_out=None, stream=None):
    """attn_fwd_kv_split for torch CUDA tensors q [B,Hq,Nq,D], k/v [B,Hkv,Nk,D].

    ``workspace``: a uint8 CUDA tensor (256-byte aligned, as torch allocates), or
    None to let torch allocate the size attn_fwd_kv_split_workspace asks for.
    Returns (o, lse) without waiting."""
    import torch

    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous [B, H, N, D]")
    o = out if out is not None else torch.empty_like(q)
    lse = None
    if with_lse:
        lse = lse_out if lse_out is not None else torch.empty((B, Hq, Nq), dtype=torch.float32,
                                                              device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if workspace is None:
        st, nbytes = attn_fwd_kv_split_workspace(B, Hq, Hkv, Nq, Nk, D, causal)
        if st != ATTN_OK:
            raise AttnError(st, "attn_fwd_kv_split_workspace")
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = attn_fwd_kv_split(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, q.dtype,
                           workspace, workspace.numel(), stream)
    if st != ATTN_OK:
        raise AttnError(st, f"attn_fwd_kv_split ({attn_last_cuda_error()})")
    return o, lse


def attn_status_str(status: int) -> str:
    return load().attn_status_str(int(status)).decode()


def attn_last_device_error(stream=None) -> int:
    return load().attn_last_device_error(_stream_handle(stream))


def attn_last_cuda_error() -> str:
    return load().attn_last_cuda_error().decode()


def attn_version() -> int:
    return load().attn_version()


def attention(q, k, v, causal: bool = True, scale: float | None = None, with_lse: bool = True,
              out=None, lse_out=None, stream=None):
    """O (and LSE) for torch CUDA tensors q [B,Hq,Nq,D], k/v [B,Hkv,Nk,D] (fp16 or bf16).

    With Nq != Nk the causal mask is bottom-right aligned (attn_fwd_kv).  torch
    allocates the outputs; the library computes them.  Launches on ``stream``
    (default: torch's current stream) and returns without waiting."""
    import torch

    B, Hq, N, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous [B, H, N, D]")
    o = out if out is not None else torch.empty_like(q)
    lse = None
    if with_lse:
        lse = lse_out if lse_out is not None else torch.empty((B, Hq, N), dtype=torch.float32,
                                                              device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if Nk == N:
        st = attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, D, scale, causal, q.dtype, stream)
    else:
        st = attn_fwd_kv(q, k, v, o, lse, B, Hq, Hkv, N, Nk, D, scale, causal, q.dtype, stream)
    if st != ATTN_OK:
        raise AttnError(st, f"attn_fwd ({attn_last_cuda_error()})")
    return o, lse
