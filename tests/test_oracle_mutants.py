"""Planted mistakes in the oracle must each break at least one pin.

Every mutant is a one-expression edit of the oracle's C source (a dropped term,
a wrong sign, index or operand), compiled on the CPU into a temporary library.
The oracle source itself stays free of test switches."""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "interleaved_groups": ("long kvh = bh / group;",
                           "long kvh = (bh / J->Hq) * J->Hkv + (bh % J->Hq) % J->Hkv;"),
    "mask_off_by_one": ("if (causal && j > i + off) {", "if (causal && j > i + off + 1) {"),
    "alignment_top_left": ("if (causal && j > i + off) {", "if (causal && j > i) {"),
    "alignment_offset_sign": ("if (causal && j > i + off) {", "if (causal && j > i - off) {"),
    "query_row_index_from_keys": ("long i = (long)(flat % J->Nq);", "long i = (long)(flat % J->Nk);"),
    "scale_dropped": ("s[j] = scale * acc;", "s[j] = acc;"),
    "max_dropped_from_lse": ("*lse_i = m + log(l);", "*lse_i = log(l);"),
    "lse_base2": ("*lse_i = m + log(l);", "*lse_i = m + log2(l);"),
    "exp_sign": ("double p = exp(s[j] - m);", "double p = exp(m - s[j]);"),
    "normalisation_dropped": ("oi[d] = oi[d] / l;", "oi[d] = oi[d];"),
    "feature_index_reversed": ("acc += qi[d] * kh[j * D + d];",
                               "acc += qi[d] * kh[j * D + (D - 1 - d)];"),
    "keys_used_as_values": ("oi[d] += s[j] * vh[j * D + d];", "oi[d] += s[j] * kh[j * D + d];"),
    "causal_mask_dropped": ("if (causal && j > i + off) {", "if (0 && j > i + off) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(before) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(before, after))
    lib = oracle.load_library(oracle.build(str(src), str(tmp_path / f"lib{name}.so")))

    def att(q, k, v, scale, causal):
        o, lse, _ = oracle.attention(q, k, v, scale, causal, nthreads=2, lib=lib)
        return o, lse

    caught = []
    for pin in ALL_PINS:
        try:
            pin(att)
        except (AssertionError, FloatingPointError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
