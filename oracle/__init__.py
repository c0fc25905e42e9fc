"""Float64 CPU oracle for the fused grouped-query attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` import this package.  The product path (the CUDA
library and its Python binding) never imports, links or calls it, and this
package never imports the product.

Two implementations of the same definition live here:

* ``attention`` / ``attention_rows`` -- the plain C routine in
  ``attn_oracle.c`` (materialised score rows in float64, mask, softmax, V
  product), multithreaded over output rows;
* ``naive.attention_naive`` -- a pure-Python triple loop for tiny inputs that
  uses the textbook formula without the max shift and exactly rounded sums.

The definition followed is the one on the page "从零开始写Qwen3"
(deepseek.csdn.net/6a3201f8..., derivation page), sections "简易情况-三矩阵相乘"
(softmax form of O) and "FlashAttention" (mask, grouped heads through
``kv_head = flattened_q_head // groups``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the C oracle with gcc (plain -O2, no fast-math) and return the .so path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11",
           *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _stale(lib_path: str) -> bool:
    return (not os.path.exists(lib_path)
            or os.path.getmtime(lib_path) < os.path.getmtime(_SRC))


def load_library(path: str | None = None):
    """Load (building first if needed) a compiled oracle and declare its C signatures."""
    global _lib
    if path is None:
        with _lock:
            if _lib is None:
                if _stale(_LIB_PATH):
                    build()
                _lib = _declare(ctypes.CDLL(_LIB_PATH))
            return _lib
    return _declare(ctypes.CDLL(path))


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_longlong)
    L = ctypes.c_long
    lib.oracle_attention.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L,
                                     ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = [dp, lp, L, dp, dp, dp, dp, L, L, L, L, L,
                                          ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_attention_kv.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L, L,
                                        ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_attention_kv.restype = ctypes.c_int
    lib.oracle_attention_rows_kv.argtypes = [dp, lp, L, dp, dp, dp, dp, L, L, L, L, L, L,
                                             ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_attention_rows_kv.restype = ctypes.c_int
    return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray, ty=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ty))


def widen(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of 16-bit storage words ("f16" or "bf16")."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def attention(q, k, v, scale: float, causal: bool, nthreads: int = 0, lib=None):
    """O [B,Hq,Nq,D] and LSE [B,Hq,Nq] (natural log) for float64 q [B,Hq,Nq,D] and
    k/v [B,Hkv,Nk,D].  With Nq != Nk the causal mask is bottom-right aligned
    (query i sees key j <= i + Nk - Nq).

    Returns (o, lse, threads_used)."""
    lib = lib or load_library()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape != (B, Hkv, Nk, D) or v.shape != k.shape:
        raise ValueError("k, v must be [B, Hkv, Nk, D] matching q")
    o = np.empty_like(q)
    lse = np.empty((B, Hq, Nq), dtype=np.float64)
    if Nq == Nk:
        rc = lib.oracle_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                  B, Hq, Hkv, Nq, D, float(scale), int(bool(causal)),
                                  int(nthreads))
    else:
        rc = lib.oracle_attention_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                     B, Hq, Hkv, Nq, Nk, D, float(scale), int(bool(causal)),
                                     int(nthreads))
    if rc <= 0:
        raise RuntimeError("oracle_attention rejected its arguments")
    return o, lse, rc


def attention_rows(q_rows, rows, k, v, Hq: int, scale: float, causal: bool,
                   nthreads: int = 0, lib=None, Nq: int | None = None):
    """Selected output rows only.

    q_rows [R, D] float64: the query row of each selected output row;
    rows [R] int: flattened (b*Hq + hq)*Nq + i; k/v [B,Hkv,Nk,D] float64;
    Nq: query rows per head (default Nk).
    Returns (o_rows [R, D], lse_rows [R], threads_used)."""
    lib = lib or load_library()
    q_rows, k, v = _f64(q_rows), _f64(k), _f64(v)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    B, Hkv, Nk, D = k.shape
    Nq = Nk if Nq is None else int(Nq)
    R = rows.shape[0]
    if q_rows.shape != (R, D):
        raise ValueError("q_rows must be [len(rows), D]")
    o = np.empty((R, D), dtype=np.float64)
    lse = np.empty((R,), dtype=np.float64)
    rc = lib.oracle_attention_rows_kv(_ptr(q_rows), _ptr(rows, ctypes.c_longlong), R,
                                      _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                      B, Hq, Hkv, Nq, Nk, D, float(scale), int(bool(causal)),
                                      int(nthreads))
    if rc <= 0:
        raise RuntimeError("oracle_attention_rows rejected its arguments")
    return o, lse, rc
