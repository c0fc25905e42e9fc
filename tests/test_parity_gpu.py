"""Parity of the CUDA path (through the C ABI) with the float64 oracle."""
import zlib

import numpy as np
import pytest

from gqa_attention_forward_gb300 import binding, workloads
from parity_util import (assert_parity, oracle_full, oracle_rows, record, run_gpu, to_device,
                         ulp_error)

pytestmark = pytest.mark.gpu


def _np(t):
    return t.double().cpu().numpy()


def _every_row(name):
    """The workload as bench.py launches it, every row of O and LSE against the oracle;
    the error is also reported in units of the storage type's ulp at |O|."""
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w)
    o, lse = run_gpu(w, x)
    og, lg = _np(o), _np(lse)
    del o, lse
    ro, rl = oracle_full(w, x)
    err = assert_parity(w, og, lg, ro, rl, name)
    ulps = ulp_error(og, ro, w.dtype)
    rows = w.B * w.Hq * w.N
    record({"workload": name, "rows": rows, "max_abs_dO": err[0], "max_rel_dLSE": err[1],
            "max_dO_ulps": ulps, "max_abs_O": float(np.max(np.abs(ro)))})
    print(f"{name}: {rows} rows max|dO|={err[0]:.3e} ({ulps:.2f} ulp) max rel dLSE={err[1]:.3e}")


@pytest.mark.parametrize("name", ["tiny_causal_gqa_f16", "pages_shape_causal_gqa_f16",
                                  "tail_stress_causal_gqa_bf16_n2000"])
def test_workload_every_row(name):
    """The small configurations and the tail/stress one (N = 2000, a ragged last tile,
    logits with std 16)."""
    _every_row(name)


@pytest.mark.parametrize("name", ["noncausal_gqa_bf16_n4096", "long_prefill_causal_gqa_bf16_n32768",
                                  "chunked_prefill_causal_gqa_bf16_q4096_k32768"])
def test_full_size_workload_every_row(name):
    """Full-size launches of the benchmarked configurations, every row against the
    float64 oracle (the long prefill takes a few minutes of the host's cores)."""
    _every_row(name)


def test_full_size_rows_spot_check():
    """A stratified row sample of the long prefill (tile boundaries, first and last
    rows) through the row entry of the oracle: the row-selection path the bench's
    CPU baseline uses agrees with the GPU on the same rows."""
    name = "long_prefill_causal_gqa_bf16_n32768"
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w)
    o, lse = run_gpu(w, x)
    rows = workloads.sample_rows(w, 600)
    og = _np(o).reshape(-1, w.D)[rows]
    lg = _np(lse).reshape(-1)[rows]
    ro, rl = oracle_rows(w, x, rows)
    assert_parity(w, og, lg, ro, rl, name)


SHAPES = [
    # B, Hq, Hkv, N, D, dtype, causal, qk_std
    (1, 1, 1, 1, 64, "f16", True, 1.0),
    (1, 1, 1, 1, 128, "bf16", False, 1.0),
    (1, 2, 1, 2, 64, "bf16", True, 1.0),
    (2, 4, 2, 63, 128, "f16", True, 1.0),
    (2, 4, 2, 63, 128, "f16", False, 1.0),
    (1, 8, 2, 127, 64, "bf16", False, 1.0),
    (1, 8, 2, 128, 128, "bf16", True, 1.0),
    (1, 4, 1, 129, 128, "f16", False, 1.0),
    (1, 4, 1, 129, 128, "bf16", True, 4.0),
    (3, 6, 3, 200, 64, "f16", True, 1.0),
    (1, 8, 8, 257, 128, "bf16", False, 4.0),
    (2, 8, 1, 384, 128, "f16", True, 1.0),
    (1, 2, 2, 1000, 64, "bf16", True, 1.0),
    (1, 16, 4, 640, 128, "bf16", False, 1.0),
    (1, 4, 4, 1024, 128, "f16", False, 1.0),
    (2, 2, 1, 1500, 64, "f16", False, 2.0),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_random_shapes(shape):
    B, Hq, Hkv, N, D, dtype, causal, std = shape
    w = workloads.Workload("rand", B, Hq, Hkv, N, D, dtype, causal, q_std=std, k_std=std,
                           seed=zlib.crc32(repr(shape).encode()) & 0xFFFF)
    x = workloads.make_inputs(w)
    o, lse = run_gpu(w, x)
    ro, rl = oracle_full(w, x)
    assert_parity(w, _np(o), _np(lse), ro, rl, str(shape))


def test_no_writes_past_the_outputs():
    """Rows >= N of the last tile are never stored: canaries after O and LSE survive."""
    import torch

    w = workloads.Workload("canary", 1, 4, 2, 200, 128, "bf16", False, seed=7)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    n_o = w.B * w.Hq * w.N * w.D
    o_buf = torch.full((n_o + 4096,), 12345.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((w.B * w.Hq * w.N + 1024,), -777.0, dtype=torch.float32, device="cuda")
    o = o_buf[:n_o].view(w.B, w.Hq, w.N, w.D)
    lse = l_buf[: w.B * w.Hq * w.N].view(w.B, w.Hq, w.N)
    binding.attention(q, k, v, causal=w.causal, scale=w.scale, out=o, lse_out=lse)
    torch.cuda.synchronize()
    assert torch.all(o_buf[n_o:] == 12345.0)
    assert torch.all(l_buf[w.B * w.Hq * w.N:] == -777.0)
    ro, rl = oracle_full(w, x)
    assert_parity(w, _np(o), _np(lse), ro, rl, "canary")


def test_lse_optional_and_deterministic():
    import torch

    w = workloads.Workload("nolse", 2, 8, 2, 300, 128, "f16", True, seed=11)
    x = workloads.make_inputs(w)
    o1, lse = run_gpu(w, x)
    o2, none = run_gpu(w, x, with_lse=False)
    assert none is None
    assert torch.equal(o1, o2)


def test_side_stream():
    import torch

    w = workloads.Workload("stream", 1, 4, 1, 256, 64, "bf16", True, seed=12)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        o, lse = binding.attention(q, k, v, causal=True, scale=w.scale, stream=s)
    assert binding.attn_last_device_error(s) == binding.ATTN_OK
    ro, rl = oracle_full(w, x)
    assert_parity(w, _np(o), _np(lse), ro, rl, "side stream")


def test_timeout_is_reported_and_context_survives():
    """A wait that nothing can satisfy runs out: the kernel records ATTN_ERR_TIMEOUT,
    drains its copies, frees TMEM and returns; the next launch is correct."""
    import torch

    lib = binding.load()
    w = workloads.Workload("stall", 1, 2, 1, 512, 128, "bf16", True, seed=13)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    try:
        lib.attn_test_set_wait_timeout_ns(300_000_000)
        lib.attn_test_inject_stall(1)
        binding.attention(q, k, v, causal=True, scale=w.scale)
        st = binding.attn_last_device_error(torch.cuda.current_stream())
    finally:
        lib.attn_test_inject_stall(0)
        lib.attn_test_set_wait_timeout_ns(0)
    assert st == binding.ATTN_ERR_TIMEOUT
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    o, lse = binding.attention(q, k, v, causal=True, scale=w.scale)
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    ro, rl = oracle_full(w, x)
    assert_parity(w, _np(o), _np(lse), ro, rl, "after timeout")


def test_scale_is_honoured():
    import torch

    from oracle import attention, widen

    w = workloads.Workload("scale", 1, 2, 1, 160, 64, "f16", False, seed=14)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o, lse = binding.attention(q, k, v, causal=False, scale=0.05)
    torch.cuda.synchronize()
    ro, rl, _ = attention(widen(x["q"], "f16"), widen(x["k"], "f16"), widen(x["v"], "f16"), 0.05, False)
    assert_parity(w, _np(o), _np(lse), ro, rl, "scale 0.05")


@pytest.mark.parametrize("name", ["pages_shape_causal_gqa_f16", "noncausal_gqa_bf16_n4096"])
def test_item_orders_give_the_same_bits(name):
    """The kv-group-major work order (a measurement hook) visits the same items with the
    same per-item arithmetic as the default order: identical O and LSE."""
    import torch

    lib = binding.load()
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w)
    o0, l0 = run_gpu(w, x)
    try:
        lib.attn_test_set_item_order(1)
        o1, l1 = run_gpu(w, x)
    finally:
        lib.attn_test_set_item_order(0)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


@pytest.fixture
def tile_kernel():
    """Selects the one-CTA-per-query-tile kernel for the test, then restores the default."""
    lib = binding.load()
    lib.attn_test_select_kernel(1)
    yield
    lib.attn_test_select_kernel(0)


@pytest.mark.parametrize("shape", SHAPES[::2], ids=lambda s: "x".join(map(str, s)))
def test_tile_kernel_random_shapes(shape, tile_kernel):
    test_random_shapes(shape)


def test_tile_kernel_timeout(tile_kernel):
    test_timeout_is_reported_and_context_survives()


def test_both_kernels_agree_on_pages_shape():
    """The two kernels compute the same function; their outputs differ by rounding only."""
    import torch

    lib = binding.load()
    w = workloads.WORKLOADS["pages_shape_causal_gqa_f16"]
    x = workloads.make_inputs(w)
    o1, l1 = run_gpu(w, x)
    try:
        lib.attn_test_select_kernel(1)
        o2, l2 = run_gpu(w, x)
    finally:
        lib.attn_test_select_kernel(0)
    assert float((o1.float() - o2.float()).abs().max()) <= 2e-3
    assert float((l1 - l2).abs().max()) <= 1e-4 * max(1.0, float(l1.abs().max()))
    assert torch.isfinite(o1).all()


# ------------------------------------------------------------------ Nq != Nk
KV_SHAPES = [
    # B, Hq, Hkv, Nq, Nk, D, dtype, causal, qk_std
    (1, 4, 2, 1, 300, 128, "bf16", True, 1.0),      # one new token over a cache
    (2, 8, 2, 7, 4096, 128, "bf16", True, 1.0),
    (2, 8, 2, 100, 1000, 128, "f16", True, 1.0),    # offset 900: two masked key tiles
    (1, 4, 4, 256, 320, 64, "bf16", True, 1.0),     # offset 64
    (1, 2, 1, 129, 256, 128, "f16", True, 1.0),     # offset 127, ragged query tile
    (1, 8, 1, 384, 385, 128, "f16", True, 1.0),     # offset 1
    (1, 2, 2, 600, 730, 128, "bf16", True, 4.0),    # near-one-hot rows
    (2, 4, 2, 300, 70, 128, "bf16", False, 1.0),    # more queries than keys, no mask
    (1, 6, 3, 90, 1000, 64, "f16", False, 2.0),
]


def _kv_workload(shape):
    B, Hq, Hkv, Nq, Nk, D, dtype, causal, std = shape
    return workloads.Workload("kv", B, Hq, Hkv, Nq, D, dtype, causal, q_std=std, k_std=std,
                              seed=zlib.crc32(repr(shape).encode()) & 0xFFFF, Nk=Nk)


@pytest.mark.parametrize("shape", KV_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_kv_shapes(shape):
    """Nq query rows over Nk keys (bottom-right causal mask), every row against the oracle."""
    w = _kv_workload(shape)
    x = workloads.make_inputs(w)
    o, lse = run_gpu(w, x)
    assert tuple(o.shape) == (w.B, w.Hq, w.N, w.D) and tuple(lse.shape) == (w.B, w.Hq, w.N)
    ro, rl = oracle_full(w, x)
    err = assert_parity(w, _np(o), _np(lse), ro, rl, str(shape))
    print(f"{shape}: max|dO|={err[0]:.3e} max rel dLSE={err[1]:.3e}")


@pytest.mark.parametrize("shape", KV_SHAPES[::2], ids=lambda s: "x".join(map(str, s)))
def test_tile_kernel_kv_shapes(shape, tile_kernel):
    test_kv_shapes(shape)


def test_kv_with_equal_lengths_is_attn_fwd():
    """attn_fwd_kv with Nq == Nk runs the same computation as attn_fwd: identical bits."""
    import torch

    w = workloads.Workload("eq", 1, 4, 2, 333, 128, "bf16", True, seed=21)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    l1 = torch.empty((1, 4, 333), dtype=torch.float32, device="cuda")
    l2 = torch.empty_like(l1)
    s = torch.cuda.current_stream()
    assert binding.attn_fwd(q, k, v, o1, l1, 1, 4, 2, 333, 128, w.scale, 1, q.dtype, s) == 0
    assert binding.attn_fwd_kv(q, k, v, o2, l2, 1, 4, 2, 333, 333, 128, w.scale, 1, q.dtype, s) == 0
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_kv_chunked_prefill_matches_one_pass():
    """Two causal chunks over a growing key prefix give the rows of one square pass
    (each within tolerance of the oracle, and of each other)."""
    import torch

    w = workloads.Workload("full", 1, 8, 2, 700, 128, "bf16", True, seed=22)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o_full, l_full = binding.attention(q, k, v, causal=True, scale=w.scale)
    cut = 300
    o_a, l_a = binding.attention(q[:, :, :cut].contiguous(), k[:, :, :cut].contiguous(),
                                 v[:, :, :cut].contiguous(), causal=True, scale=w.scale)
    o_b, l_b = binding.attention(q[:, :, cut:].contiguous(), k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    o_cat = torch.cat([o_a, o_b], dim=2)
    l_cat = torch.cat([l_a, l_b], dim=2)
    ro, rl = oracle_full(w, x)
    assert_parity(w, _np(o_cat), _np(l_cat), ro, rl, "chunked")
    assert float((o_cat.float() - o_full.float()).abs().max()) <= 1.6e-2



def test_cuda_graph_capture_and_replay():
    """A call captured into a CUDA graph replays correctly, also on new inputs copied
    into the captured buffers; replays keep working after an error was reported."""
    import torch

    w = workloads.WORKLOADS["pages_shape_causal_gqa_f16"]
    x1 = workloads.make_inputs(w)
    x2 = workloads.make_inputs(w, seed=w.seed + 100)
    q, k, v = (to_device(x1[n], w.dtype) for n in "qkv")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device="cuda")
    binding.attention(q, k, v, causal=True, scale=w.scale, out=o, lse_out=lse)  # first use
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.attention(q, k, v, causal=True, scale=w.scale, out=o, lse_out=lse)
    o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    ro, rl = oracle_full(w, x1)
    assert_parity(w, _np(o), _np(lse), ro, rl, "graph replay")
    for name, t in zip("qkv", (q, k, v)):
        t.copy_(to_device(x2[name], w.dtype))
    graph.replay()
    graph.replay()
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    ro2, rl2 = oracle_full(w, x2)
    assert_parity(w, _np(o), _np(lse), ro2, rl2, "graph replay, new inputs")


# ------------------------------------------------------------------ packed short queries
DECODE_SHAPES = [
    # B, Hq, Hkv, Nq, Nk, D, dtype, causal, qk_std, forced splits (0 = chosen)
    (1, 32, 8, 1, 4096, 128, "bf16", True, 1.0, 0),     # one token over a cache
    (2, 8, 2, 1, 1000, 128, "f16", True, 1.0, 3),       # ragged key tail
    (1, 8, 1, 16, 3000, 128, "bf16", True, 1.0, 5),     # 8 heads x 16 rows = one full tile
    (2, 4, 2, 7, 700, 64, "f16", True, 2.0, 0),
    (1, 16, 2, 40, 900, 128, "bf16", True, 1.0, 4),     # 320 rows: tiles cut rows of a head
    (1, 4, 4, 100, 100, 128, "bf16", True, 1.0, 2),     # square: some splits see no key
    (1, 8, 2, 5, 2000, 128, "bf16", False, 1.0, 0),     # no mask
    (2, 4, 1, 3, 520, 128, "bf16", True, 4.0, 3),       # near-one-hot rows
    (1, 2, 1, 1, 1, 64, "f16", True, 1.0, 0),
    (1, 8, 2, 2, 6000, 128, "bf16", True, 1.0, 47),    # 47 pieces: three merge batches
]


@pytest.fixture
def forced_splits():
    lib = binding.load()
    yield lib.attn_test_force_splits
    lib.attn_test_force_splits(0)


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_decode_shapes(shape, forced_splits):
    """attn_fwd_decode (grouped-query packing, key splits and their merge): every row
    against the oracle."""
    import torch

    B, Hq, Hkv, Nq, Nk, D, dtype, causal, std, splits = shape
    forced_splits(splits)
    w = workloads.Workload("dec", B, Hq, Hkv, Nq, D, dtype, causal, q_std=std, k_std=std,
                           seed=zlib.crc32(repr(shape).encode()) & 0xFFFF, Nk=Nk)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    o, lse = binding.attention_decode(q, k, v, causal=causal, scale=w.scale, workspace=ws)
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    ro, rl = oracle_full(w, x)
    err = assert_parity(w, _np(o), _np(lse), ro, rl, str(shape))
    print(f"{shape}: max|dO|={err[0]:.3e} max rel dLSE={err[1]:.3e}")


def test_decode_without_workspace_and_sizes():
    """No workspace: one split, same function.  The size query asks for room for
    several splits when few kv heads are in play, none when the row tiles fill the GPU."""
    import torch

    st, nbytes = binding.attn_fwd_decode_workspace(1, 32, 8, 1, 32768, 128)
    assert st == binding.ATTN_OK and nbytes > 0
    st, big = binding.attn_fwd_decode_workspace(512, 32, 8, 1, 4096, 128)
    assert st == binding.ATTN_OK and big == 0
    w = workloads.Workload("dec0", 1, 8, 2, 3, 128, "bf16", True, seed=31, Nk=1500)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o = torch.empty_like(q)
    lse = torch.empty((1, 8, 3), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    assert binding.attn_fwd_decode(q, k, v, o, lse, 1, 8, 2, 3, 1500, 128, w.scale, 1, q.dtype,
                                   None, 0, s) == binding.ATTN_OK
    assert binding.attn_last_device_error(s) == binding.ATTN_OK
    ro, rl = oracle_full(w, x)
    assert_parity(w, _np(o), _np(lse), ro, rl, "one split")


def test_decode_agrees_with_kv_path():
    """The packed kernel and the general kernel compute the same function."""
    w = workloads.Workload("deckv", 2, 16, 4, 9, 128, "bf16", True, seed=32, Nk=2500)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o1, l1 = binding.attention(q, k, v, causal=True, scale=w.scale)
    o2, l2 = binding.attention_decode(q, k, v, causal=True, scale=w.scale)
    import torch

    torch.cuda.synchronize()
    assert float((o1.float() - o2.float()).abs().max()) <= 1.6e-2
    assert float(((l1 - l2).abs() / l1.abs().clamp_min(1.0)).max()) <= 1e-4


def test_decode_timeout_is_reported_and_context_survives(forced_splits):
    """The packed split kernel under a wait nothing satisfies (the Q load is skipped):
    it records ATTN_ERR_TIMEOUT and returns; the next call is correct."""
    import torch

    lib = binding.load()
    forced_splits(4)
    w = workloads.Workload("dstall", 1, 8, 2, 2, 128, "bf16", True, seed=33, Nk=1500)
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    ws = torch.empty(8 << 20, dtype=torch.uint8, device="cuda")
    try:
        lib.attn_test_set_wait_timeout_ns(300_000_000)
        lib.attn_test_inject_stall(1)
        binding.attention_decode(q, k, v, causal=True, scale=w.scale, workspace=ws)
        st = binding.attn_last_device_error(torch.cuda.current_stream())
    finally:
        lib.attn_test_inject_stall(0)
        lib.attn_test_set_wait_timeout_ns(0)
    assert st == binding.ATTN_ERR_TIMEOUT
    o, lse = binding.attention_decode(q, k, v, causal=True, scale=w.scale, workspace=ws)
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    ro, rl = oracle_full(w, x)
    assert_parity(w, _np(o), _np(lse), ro, rl, "decode after timeout")


def test_decode_repeated_calls_and_graph_replays(forced_splits):
    """The split kernel and the merge kernel of attn_fwd_decode (programmatic dependent
    launches): one workspace, calls in a row with new inputs, then a captured call
    replayed twice on new inputs."""
    import torch

    forced_splits(6)
    w = workloads.Workload("drep", 2, 16, 4, 5, 128, "bf16", True, seed=34, Nk=3000)
    st, nbytes = binding.attn_fwd_decode_workspace(w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D)
    assert st == binding.ATTN_OK and nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    xs = [workloads.make_inputs(w, seed=w.seed + t) for t in range(4)]
    q, k, v = (to_device(xs[0][n], w.dtype) for n in "qkv")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device="cuda")

    def call():  # on torch's current stream (the capture stream inside the graph block)
        assert binding.attn_fwd_decode(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D, w.scale,
                                       1, q.dtype, ws, ws.numel(),
                                       torch.cuda.current_stream()) == binding.ATTN_OK

    def check(x, what):
        torch.cuda.synchronize()
        assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
        ro, rl = oracle_full(w, x)
        assert_parity(w, _np(o), _np(lse), ro, rl, what)

    for t in range(2):
        for name, tt in zip("qkv", (q, k, v)):
            tt.copy_(to_device(xs[t][name], w.dtype))
        call()
        check(xs[t], f"call {t}")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for t in (2, 3):
        for name, tt in zip("qkv", (q, k, v)):
            tt.copy_(to_device(xs[t][name], w.dtype))
        graph.replay()
        check(xs[t], f"replay {t}")


# ------------------------------------------------------------------ host buffers
def _host_call(w, x, pinned=True):
    """attn_fwd_host on host copies of the inputs; returns (o, lse) as host tensors and
    the device outputs."""
    import torch

    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16

    def host(bits):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(dt)
        return t.pin_memory() if pinned else t.clone()

    qh, kh, vh = (host(x[n]) for n in "qkv")
    oh = torch.empty_like(qh)
    lh = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32)
    if pinned:
        oh, lh = oh.pin_memory(), lh.pin_memory()
    qd, kd, vd = (torch.empty(t.shape, dtype=dt, device="cuda") for t in (qh, kh, vh))
    od = torch.empty_like(qd)
    ld = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    st = binding.attn_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, w.B, w.Hq, w.Hkv, w.N,
                               w.n_keys, w.D, w.scale, w.causal, dt, s)
    assert st == binding.ATTN_OK, binding.STATUS.get(st, st)
    s.synchronize()
    assert binding.attn_last_device_error(s) == binding.ATTN_OK
    return oh, lh, od, ld


@pytest.mark.parametrize("name", ["long_prefill_causal_gqa_bf16_n32768", "noncausal_gqa_bf16_n4096"])
def test_host_buffers_same_bits_as_device_call(name):
    """Chunked copies and compute give the same bits as one device-resident call
    (each row's arithmetic does not depend on the chunking)."""
    import torch

    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w)
    oh, lh, od, ld = _host_call(w, x)
    o, lse = run_gpu(w, x)
    assert torch.equal(oh, o.cpu()) and torch.equal(lh, lse.cpu())
    assert torch.equal(od.cpu(), oh)


@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffers_against_oracle(pinned):
    w = workloads.Workload("host", 3, 8, 2, 200, 128, "bf16", True, seed=51, Nk=700)
    x = workloads.make_inputs(w)
    oh, lh, _, _ = _host_call(w, x, pinned=pinned)
    ro, rl = oracle_full(w, x)
    assert_parity(w, oh.double().numpy(), lh.double().numpy(), ro, rl, f"host pinned={pinned}")


@pytest.mark.parametrize("name", ["decode_gqa_bf16_b1_q1_k32768", "decode_gqa_bf16_b16_q1_k8192",
                                  "short_chunk_gqa_bf16_q16_k32768"])
def test_decode_workloads_full_size(name):
    """The benchmarked decode workloads, as bench.py runs them (attn_fwd_decode with the
    workspace it asks for): every row against the oracle."""
    import torch

    w = workloads.WORKLOADS[name]
    assert w.entry == "attn_fwd_decode"
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o, lse = binding.attention_decode(q, k, v, causal=w.causal, scale=w.scale)
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    ro, rl = oracle_full(w, x)
    err = assert_parity(w, _np(o), _np(lse), ro, rl, name)
    print(f"{name}: max|dO|={err[0]:.3e} max rel dLSE={err[1]:.3e}")


# ------------------------------------------------------------------ randomized sweep
def _random_problems(count=24, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for t in range(count):
        B = int(rng.integers(1, 4))
        Hkv = int(rng.choice([1, 2, 4]))
        G = int(rng.choice([1, 2, 4, 8]))
        causal = bool(rng.integers(0, 2))
        Nq = int(rng.integers(1, 300))
        Nk = int(rng.integers(Nq, 1500)) if causal else int(rng.integers(1, 1500))
        D = int(rng.choice([64, 128]))
        dtype = str(rng.choice(["f16", "bf16"]))
        std = float(rng.choice([1.0, 3.0]))
        out.append((t, B, G * Hkv, Hkv, Nq, Nk, D, dtype, causal, std))
    return out


@pytest.mark.parametrize("prob", _random_problems(), ids=lambda p: "x".join(map(str, p)))
def test_random_problems_all_entry_points(prob):
    """Seeded random problems through attn_fwd_kv, attn_fwd_decode, attn_fwd_host and
    attn_fwd_kv_split (which cuts the last round into key ranges when it can), each
    against the oracle."""
    import torch

    t, B, Hq, Hkv, Nq, Nk, D, dtype, causal, std = prob
    w = workloads.Workload("fuzz", B, Hq, Hkv, Nq, D, dtype, causal, q_std=std, k_std=std,
                           seed=3000 + t, Nk=Nk)
    x = workloads.make_inputs(w)
    ro, rl = oracle_full(w, x)
    q, k, v = (to_device(x[n], dtype) for n in "qkv")
    o1, l1 = binding.attention(q, k, v, causal=causal, scale=w.scale)
    o2, l2 = binding.attention_decode(q, k, v, causal=causal, scale=w.scale)
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    assert_parity(w, _np(o1), _np(l1), ro, rl, f"{prob} attn_fwd_kv")
    assert_parity(w, _np(o2), _np(l2), ro, rl, f"{prob} attn_fwd_decode")
    oh, lh, _, _ = _host_call(w, x)
    assert_parity(w, oh.double().numpy(), lh.double().numpy(), ro, rl, f"{prob} attn_fwd_host")
    o3, l3 = binding.attention_split(q, k, v, causal=causal, scale=w.scale)
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    assert_parity(w, _np(o3), _np(l3), ro, rl, f"{prob} attn_fwd_kv_split")


# ------------------------------------------------------------------ key-split last round
SPLIT_SHAPES = [
    # B, Hq, Hkv, Nq, Nk, D, dtype, causal, qk_std: few enough equal-length items that
    # the plan cuts the last (here: only) round into key ranges
    (1, 4, 2, 3000, 3000, 128, "bf16", False, 1.0),   # 48 items, ragged keys
    (1, 8, 2, 700, 9000, 128, "bf16", True, 1.0),     # a chunk over a longer cache
    (2, 2, 1, 1000, 1000, 64, "f16", False, 2.0),
    (1, 4, 4, 300, 5000, 128, "f16", True, 4.0),      # near-one-hot rows, causal offset 4700
    (1, 2, 1, 129, 2000, 128, "bf16", True, 1.0),     # ragged query tile
]


def _split_workload(shape):
    B, Hq, Hkv, Nq, Nk, D, dtype, causal, std = shape
    return workloads.Workload("split", B, Hq, Hkv, Nq, D, dtype, causal, q_std=std, k_std=std,
                              seed=zlib.crc32(repr(shape).encode()) & 0xFFFF, Nk=Nk)


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_split_shapes(shape):
    """attn_fwd_kv_split cuts these items into key ranges and merges the pieces: every row
    against the oracle, and within tolerance of the uncut call."""
    import torch

    w = _split_workload(shape)
    st, nbytes = binding.attn_fwd_kv_split_workspace(w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D, w.causal)
    assert st == binding.ATTN_OK and nbytes > 0, "the plan should cut this problem"
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o, lse = binding.attention_split(q, k, v, causal=w.causal, scale=w.scale)
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    ro, rl = oracle_full(w, x)
    err = assert_parity(w, _np(o), _np(lse), ro, rl, str(shape))
    o2, l2 = binding.attention(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert float((o.float() - o2.float()).abs().max()) <= (2e-3 if w.dtype == "f16" else 1.6e-2)
    assert float(((lse - l2).abs() / l2.abs().clamp_min(1.0)).max()) <= 1e-4
    print(f"{shape}: max|dO|={err[0]:.3e} max rel dLSE={err[1]:.3e}")


def test_split_workspace_sizes():
    """Causal problems with Nq == Nk are not cut (their items already differ in length);
    a problem that fills many rounds exactly is not cut either."""
    st, n = binding.attn_fwd_kv_split_workspace(1, 32, 8, 32768, 32768, 128, True)
    assert st == binding.ATTN_OK and n == 0
    st, n = binding.attn_fwd_kv_split_workspace(4, 32, 8, 4096, 4096, 128, False)
    assert st == binding.ATTN_OK and n > 0  # 2048 items: the 14th round holds 72


def test_split_repeated_calls_and_graph_replays():
    """One workspace, calls in a row with new inputs, then a captured call replayed twice on
    new inputs (the arrival counters carry the launch's sequence number, and the last
    arrival leaves them at zero for the next replay)."""
    import torch

    w = _split_workload(SPLIT_SHAPES[0])
    st, nbytes = binding.attn_fwd_kv_split_workspace(w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D, w.causal)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    xs = [workloads.make_inputs(w, seed=w.seed + t) for t in range(4)]
    q, k, v = (to_device(xs[0][n], w.dtype) for n in "qkv")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device="cuda")

    def call():
        binding.attention_split(q, k, v, causal=w.causal, scale=w.scale, workspace=ws, out=o,
                                lse_out=lse)

    def check(x, what):
        torch.cuda.synchronize()
        assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
        ro, rl = oracle_full(w, x)
        assert_parity(w, _np(o), _np(lse), ro, rl, what)

    for t in range(2):
        for name, tt in zip("qkv", (q, k, v)):
            tt.copy_(to_device(xs[t][name], w.dtype))
        call()
        check(xs[t], f"call {t}")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for t in (2, 3):
        for name, tt in zip("qkv", (q, k, v)):
            tt.copy_(to_device(xs[t][name], w.dtype))
        graph.replay()
        check(xs[t], f"replay {t}")


def test_split_timeout_is_reported_and_context_survives():
    """The split path under a wait nothing satisfies: ATTN_ERR_TIMEOUT, and the next call
    (new launch sequence number, same workspace) is correct."""
    import torch

    lib = binding.load()
    w = _split_workload(SPLIT_SHAPES[2])
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    st, nbytes = binding.attn_fwd_kv_split_workspace(w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D, w.causal)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    try:
        lib.attn_test_set_wait_timeout_ns(300_000_000)
        lib.attn_test_inject_stall(1)
        binding.attention_split(q, k, v, causal=w.causal, scale=w.scale, workspace=ws)
        st = binding.attn_last_device_error(torch.cuda.current_stream())
    finally:
        lib.attn_test_inject_stall(0)
        lib.attn_test_set_wait_timeout_ns(0)
    assert st == binding.ATTN_ERR_TIMEOUT
    o, lse = binding.attention_split(q, k, v, causal=w.causal, scale=w.scale, workspace=ws)
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    ro, rl = oracle_full(w, x)
    assert_parity(w, _np(o), _np(lse), ro, rl, "split after timeout")


@pytest.mark.parametrize("name", ["noncausal_gqa_bf16_n4096", "chunked_prefill_causal_gqa_bf16_q4096_k32768"])
def test_split_full_size_every_row(name):
    """The two equal-length benchmark workloads through attn_fwd_kv_split (their last
    round is cut in two): every row against the oracle."""
    import torch

    w = workloads.WORKLOADS[name]
    st, nbytes = binding.attn_fwd_kv_split_workspace(w.B, w.Hq, w.Hkv, w.N, w.n_keys, w.D, w.causal)
    assert st == binding.ATTN_OK and nbytes > 0
    x = workloads.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in "qkv")
    o, lse = binding.attention_split(q, k, v, causal=w.causal, scale=w.scale)
    assert binding.attn_last_device_error(torch.cuda.current_stream()) == binding.ATTN_OK
    og, lg = _np(o), _np(lse)
    del o, lse
    ro, rl = oracle_full(w, x)
    err = assert_parity(w, og, lg, ro, rl, name + " split")
    record({"workload": name + " (attn_fwd_kv_split)", "rows": w.B * w.Hq * w.N, "max_abs_dO": err[0],
            "max_rel_dLSE": err[1], "max_dO_ulps": ulp_error(og, ro, w.dtype)})
