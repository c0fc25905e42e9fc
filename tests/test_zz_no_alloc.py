"""attn_fwd_decode_noalloc: the packed, key-split kernel with the library's fixed
device scratch instead of a caller workspace.

It must give the same bits as attn_fwd_decode (same split plan, same kernels) on
two calls in a row with different inputs, match the oracle, and refuse a plan that
needs more scratch than the buffer holds without touching the outputs.  The file
is collected last and also runs on its own (its first call then does the one-time
lookup of the buffer's address)."""
import numpy as np
import pytest

from gqa_attention_forward_gb300 import binding, workloads
from parity_util import assert_parity, oracle_full, to_device

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, Hq, Hkv, Nq, Nk, D, dtype, causal
    (1, 32, 8, 1, 32768, 128, "bf16", True),   # one token over a long cache: many splits
    (1, 32, 8, 16, 4096, 128, "f16", True),
    (2, 8, 2, 3, 1500, 64, "bf16", False),
]


def _outputs(torch, w):
    o = torch.empty((w.B, w.Hq, w.N, w.D), dtype=torch.float16 if w.dtype == "f16" else torch.bfloat16,
                    device="cuda")
    return o, torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_same_bits_as_the_workspace_entry_on_two_calls(shape):
    import torch

    B, Hq, Hkv, Nq, Nk, D, dtype, causal = shape
    w = workloads.Workload("na", B, Hq, Hkv, Nq, D, dtype, causal, seed=41, Nk=Nk)
    st, nbytes = binding.attn_fwd_decode_workspace(B, Hq, Hkv, Nq, Nk, D)
    assert st == binding.ATTN_OK and nbytes <= 16 << 20
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    for call in range(2):
        x = workloads.make_inputs(w, seed=w.seed + call)
        q, k, v = (to_device(x[n], dtype) for n in "qkv")
        o1, l1 = _outputs(torch, w)
        o2, l2 = _outputs(torch, w)
        args = (B, Hq, Hkv, Nq, Nk, D, w.scale, causal, q.dtype)
        assert binding.attn_fwd_decode(q, k, v, o1, l1, *args, ws, ws.numel(), s) == binding.ATTN_OK
        assert binding.attn_fwd_decode_noalloc(q, k, v, o2, l2, *args, s) == binding.ATTN_OK
        assert binding.attn_last_device_error(s) == binding.ATTN_OK
        assert torch.equal(o1, o2), f"call {call}: O differs"
        assert torch.equal(l1, l2), f"call {call}: LSE differs"
        assert torch.isfinite(o2.float()).all() and torch.isfinite(l2).all()


def test_matches_the_oracle():
    import torch

    w = workloads.Workload("na_or", 1, 8, 2, 4, 128, "bf16", True, seed=42, Nk=2900)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o, lse = _outputs(torch, w)
    s = torch.cuda.current_stream()
    st = binding.attn_fwd_decode_noalloc(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D,
                                         w.scale, True, q.dtype, s)
    assert st == binding.ATTN_OK
    assert binding.attn_last_device_error(s) == binding.ATTN_OK
    ro, rl = oracle_full(w, x)
    assert_parity(w, o.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "no-alloc")


def test_refuses_a_plan_larger_than_the_buffer():
    """64 forced splits of 512 rows need 64 * 512 * 129 * 4 B > 16 MiB: refused before
    any launch, outputs untouched; the next call with the chosen plan works."""
    import torch

    lib = binding.load()
    w = workloads.Workload("na_big", 1, 32, 8, 16, 128, "bf16", True, seed=43, Nk=32768)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o, lse = _outputs(torch, w)
    o.fill_(3.0)
    lse.fill_(-5.0)
    s = torch.cuda.current_stream()
    args = (w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D, w.scale, True, q.dtype)
    try:
        lib.attn_test_force_splits(64)
        st = binding.attn_fwd_decode_noalloc(q, k, v, o, lse, *args, s)
    finally:
        lib.attn_test_force_splits(0)
    assert st == binding.ATTN_ERR_SCRATCH
    assert binding.attn_status_str(st) != "unknown status"
    torch.cuda.synchronize()
    assert bool((o == 3.0).all()) and bool((lse == -5.0).all())
    assert binding.attn_fwd_decode_noalloc(q, k, v, o, lse, *args, s) == binding.ATTN_OK
    assert binding.attn_last_device_error(s) == binding.ATTN_OK
    assert torch.isfinite(lse).all()
