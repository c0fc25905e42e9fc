"""The float64 oracle against its pins (closed forms, invariants, library routines,
brute force), plus consistency of its row-sampled entry point."""
import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS


def _att(q, k, v, scale, causal):
    o, lse, _ = oracle.attention(q, k, v, scale, causal, nthreads=2)
    return o, lse


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(_att)


def test_rows_entry_matches_full():
    rng = np.random.default_rng(0)
    B, Hq, Hkv, N, D = 2, 4, 2, 70, 16
    q = rng.standard_normal((B, Hq, N, D))
    k = rng.standard_normal((B, Hkv, N, D))
    v = rng.standard_normal((B, Hkv, N, D))
    for causal in (True, False):
        o, lse, _ = oracle.attention(q, k, v, 0.25, causal)
        rows = np.array([0, 1, 69, 70, 139, 200, 559], dtype=np.int64)
        q_rows = q.reshape(-1, D)[rows]
        orow, lrow, _ = oracle.attention_rows(q_rows, rows, k, v, Hq, 0.25, causal)
        assert np.array_equal(orow, o.reshape(-1, D)[rows])
        assert np.array_equal(lrow, lse.reshape(-1)[rows])


def test_thread_count_does_not_change_result():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 2, 50, 8))
    k = rng.standard_normal((1, 1, 50, 8))
    v = rng.standard_normal((1, 1, 50, 8))
    a = oracle.attention(q, k, v, 0.3, True, nthreads=1)
    b = oracle.attention(q, k, v, 0.3, True, nthreads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert a[2] == 1 and b[2] == 7


def test_rejects_bad_grouping():
    q = np.zeros((1, 3, 4, 8))
    k = np.zeros((1, 2, 4, 8))
    with pytest.raises(RuntimeError):
        oracle.attention(q, k, k, 1.0, True)
