"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the float64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
from gqa_attention_forward_gb300 import binding, workloads

# Tolerances stated for this operation: O max |err| 2e-3 (fp16) / 1.6e-2 (bf16);
# LSE |err| <= 1e-4 * max(1, |LSE|) (relative, floored at 1 because LSE can be ~0).
O_TOL = {"f16": 2e-3, "bf16": 1.6e-2}
LSE_RTOL = 1e-4


def to_device(bits: np.ndarray, dtype: str):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16).cuda()


def run_gpu(w: workloads.Workload, x: dict, with_lse: bool = True):
    import torch

    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o, lse = binding.attention(q, k, v, causal=w.causal, scale=w.scale, with_lse=with_lse)
    st = binding.attn_last_device_error(torch.cuda.current_stream())
    assert st == binding.ATTN_OK, f"device error {binding.STATUS.get(st, st)}"
    return o, lse


def oracle_full(w: workloads.Workload, x: dict):
    o, lse, _ = oracle.attention(oracle.widen(x["q"], w.dtype), oracle.widen(x["k"], w.dtype),
                                 oracle.widen(x["v"], w.dtype), w.scale, w.causal)
    return o, lse


def oracle_rows(w: workloads.Workload, x: dict, rows: np.ndarray):
    q_rows = oracle.widen(x["q"].reshape(-1, w.D)[rows], w.dtype)
    o, lse, _ = oracle.attention_rows(q_rows, rows, oracle.widen(x["k"], w.dtype),
                                      oracle.widen(x["v"], w.dtype), w.Hq, w.scale, w.causal,
                                      Nq=w.N)
    return o, lse


def errors(o_gpu: np.ndarray, lse_gpu, o_ref: np.ndarray, lse_ref):
    err_o = float(np.max(np.abs(o_gpu - o_ref))) if o_ref.size else 0.0
    err_lse = 0.0
    if lse_gpu is not None and lse_ref.size:
        err_lse = float(np.max(np.abs(lse_gpu - lse_ref) / np.maximum(1.0, np.abs(lse_ref))))
    return err_o, err_lse


# Significand bits after the leading one: the spacing of representable values
# in [2^e, 2^(e+1)) is 2^(e - bits); below the smallest normal the spacing stays
# that of the smallest normal binade.
_FRAC_BITS = {"bf16": 7, "f16": 10}
_MIN_EXP = {"bf16": -126, "f16": -14}


def ulp_of(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the 16-bit storage type's values at |x| (one unit in the last place)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, np.finfo(np.float64).tiny)))
    e = np.maximum(e, _MIN_EXP[dtype])
    return np.exp2(e - _FRAC_BITS[dtype])


def ulp_error(o_gpu: np.ndarray, o_ref: np.ndarray, dtype: str, floor: float = 1.0) -> float:
    """max over elements of |O_gpu - O_ref| in units of the storage type's ulp at
    max(|O_ref|, floor).  The floor (1 by default, the same floor as the LSE
    tolerance) keeps outputs near zero, whose own ulp is tiny while their error is
    set by the scale of V, from dominating the figure."""
    if o_ref.size == 0:
        return 0.0
    scale = np.maximum(np.abs(o_ref), floor)
    return float(np.max(np.abs(o_gpu - o_ref) / ulp_of(scale, dtype)))


def record(entry: dict) -> None:
    """Append one parity result to the JSON-lines file named by GQA_PARITY_LOG, if set."""
    path = os.environ.get("GQA_PARITY_LOG")
    if path:
        with open(path, "a") as fh:
            fh.write(json.dumps(entry) + "\n")


def assert_parity(w, o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    if lse_gpu is not None:
        assert np.all(np.isfinite(lse_gpu)), f"{what}: non-finite LSE"
    err_o, err_lse = errors(o_gpu, lse_gpu, o_ref, lse_ref)
    assert err_o <= O_TOL[w.dtype], f"{what}: max|dO| {err_o:.3e} > {O_TOL[w.dtype]:.1e}"
    assert err_lse <= LSE_RTOL, f"{what}: max rel dLSE {err_lse:.3e} > {LSE_RTOL:.1e}"
    return err_o, err_lse
