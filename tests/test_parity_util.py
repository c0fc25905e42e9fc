"""The ulp measure the GPU parity tests report, checked against the storage
formats' definitions (CPU)."""
import numpy as np

from parity_util import ulp_error, ulp_of


def test_ulp_of_bf16_binades():
    # bfloat16 keeps 8 significant bits: spacing 2^(e-7) in [2^e, 2^(e+1))
    assert ulp_of(np.array([1.0]), "bf16")[0] == 2.0 ** -7
    assert ulp_of(np.array([1.99]), "bf16")[0] == 2.0 ** -7
    assert ulp_of(np.array([-4.5]), "bf16")[0] == 2.0 ** -5
    assert ulp_of(np.array([0.3]), "bf16")[0] == 2.0 ** -9
    assert ulp_of(np.array([0.0]), "bf16")[0] == 2.0 ** -133


def test_ulp_of_f16_binades_and_subnormals():
    # binary16 keeps 11 significant bits; below 2^-14 the spacing stays 2^-24
    assert ulp_of(np.array([1.0]), "f16")[0] == 2.0 ** -10
    assert ulp_of(np.array([1000.0]), "f16")[0] == 0.5
    assert ulp_of(np.array([2.0 ** -20]), "f16")[0] == 2.0 ** -24
    assert ulp_of(np.array([0.0]), "f16")[0] == 2.0 ** -24


def test_ulp_matches_numpy_float16_spacing():
    x = np.array([0.001, 0.5, 3.0, 700.0, -12.25])
    assert np.array_equal(ulp_of(x, "f16"), np.abs(np.spacing(x.astype(np.float16))).astype(np.float64))


def test_ulp_error_is_in_units_of_the_reference():
    ref = np.array([4.0, 1.0, -0.25])
    got = ref + np.array([2.0 ** -5, 0.0, 0.0])  # one bf16 ulp at 4
    assert ulp_error(got, ref, "bf16") == 1.0


def test_ulp_error_floors_small_outputs_at_one():
    ref = np.array([1e-3, 2.0])
    got = ref + np.array([2.0 ** -7, 0.0])  # one bf16 ulp of 1 on a tiny output
    assert ulp_error(got, ref, "bf16") == 1.0
    assert ulp_error(got, ref, "bf16", floor=0.0) > 100
