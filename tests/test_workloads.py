"""The shared seeded input generator: rounding, determinism, distributions."""
import numpy as np

import oracle
from gqa_attention_forward_gb300 import workloads as W


def test_bf16_rounding_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 1.0 + 2.0 ** -9,
                  65504.0, 3.0e38], dtype=np.float32)
    bits = W.f32_to_bf16_bits(x)
    # 1+2^-8 is a tie -> even (1.0); 1+3*2^-8 is a tie -> even (1+2^-6... i.e. 0x3F82)
    assert bits.tolist()[:5] == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F80]
    back = oracle.widen(bits, "bf16")
    assert back[0] == 1.0 and back[3] == -2.5
    assert np.all(np.abs(back - x.astype(np.float64)) <= np.abs(x) * 2.0 ** -8)


def test_f16_rounding_roundtrip():
    x = np.array([0.1, -3.75, 1.0 / 3.0, 1e-5], dtype=np.float32)
    bits = W.f32_to_f16_bits(x)
    assert np.array_equal(oracle.widen(bits, "f16"), x.astype(np.float16).astype(np.float64))


def test_inputs_deterministic_and_shaped():
    w = W.WORKLOADS["tiny_causal_gqa_f16"]
    a, b = W.make_inputs(w), W.make_inputs(w)
    for n in "qkv":
        assert np.array_equal(a[n], b[n])
        assert a[n].dtype == np.uint16
    assert a["q"].shape == (1, 2, 128, 64) and a["k"].shape == (1, 1, 128, 64)
    c = W.make_inputs(w, seed=w.seed + 1)
    assert not np.array_equal(a["q"], c["q"])


def test_stress_distribution():
    w = W.WORKLOADS["tail_stress_causal_gqa_bf16_n2000"].with_(B=1, Hq=8, Hkv=1, N=500)
    x = W.make_inputs(w)
    q = oracle.widen(x["q"], "bf16")
    v = oracle.widen(x["v"], "bf16")
    assert abs(q.std() - 4.0) < 0.05 and abs(v.std() - 1.0) < 0.02
    assert abs(q.mean()) < 0.05


def test_workload_table_matches_flop_convention():
    w = W.WORKLOADS["long_prefill_causal_gqa_bf16_n32768"]
    assert w.flops == 2.0 * 1 * 32 * 32768 ** 2 * 128
    w3 = W.WORKLOADS["noncausal_gqa_bf16_n4096"]
    assert w3.flops == 4.0 * 4 * 32 * 4096 ** 2 * 128
    for w in W.WORKLOADS.values():
        assert w.Hq % w.Hkv == 0


def test_sample_rows_cover_edges():
    w = W.WORKLOADS["tail_stress_causal_gqa_bf16_n2000"]
    rows = W.sample_rows(w, 600)
    assert rows.min() >= 0 and rows.max() < w.B * w.Hq * w.N
    i = rows % w.N
    assert {0, 127, 128, 1999}.issubset(set(i.tolist()))
