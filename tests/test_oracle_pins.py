"""The fp64 oracle against its pins (no GPU)."""
import numpy as np
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_mod):
    pin(oracle_mod.default())


def test_golden_numbers_match_their_closed_forms():
    P.pin_golden_derivations()


def test_out_of_range_slot_is_rejected(oracle_mod):
    q, k, v, indptr, indices, scale = P.random_case(np.random.default_rng(0), [3], 4, 2, 8)
    bad = indices.copy()
    bad[1] = k.shape[0]
    with pytest.raises(ValueError):
        oracle_mod.decode(q, k, v, indptr, bad, 4, 2, 8, scale)
    with pytest.raises(ValueError):
        oracle_mod.append(k, np.array([k.shape[0]], np.int32), k[:1])


def test_thread_count_does_not_change_results(oracle_mod):
    rng = np.random.default_rng(11)
    q, k, v, indptr, indices, scale = P.random_case(rng, [100, 3, 57, 9], 32, 8, 128)
    a = oracle_mod.decode(q, k, v, indptr, indices, 32, 8, 128, scale, n_threads=1)
    b = oracle_mod.decode(q, k, v, indptr, indices, 32, 8, 128, scale, n_threads=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_prefill_rejects_chunk_longer_than_context(oracle_mod):
    rng = np.random.default_rng(3)
    q, k, v, qo, kvp, idx, scale = P.prefill_case(rng, [2], [2], 2, 1, 4)
    with pytest.raises(ValueError):
        oracle_mod.prefill(q, k, v, np.array([0, 2], np.int32), np.array([0, 1], np.int32),
                           idx[:1], 2, 1, 4, scale)
