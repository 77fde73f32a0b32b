"""Host round driver (spec_round_update, C ABI, no GPU) against the oracle's
round bookkeeping, on random round streams and on inconsistent states."""
import ctypes

import numpy as np
import pytest

import oracle
import speculative_decoding_verification_54_gb300 as sv
from speculative_decoding_verification_54_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sv.load()


def _states(rows):
    arr = (sv.SpecRoundState * len(rows))()
    for i, (g, s, k) in enumerate(rows):
        arr[i].gamma, arr[i].seq_len, arr[i].kv_len = g, s, k
    return arr


def test_round_driver_matches_the_oracle(lib):
    rng = np.random.default_rng(17)
    B = 37
    init = [(int(rng.integers(1, 9)), int(s), int(s) - 1) for s in rng.integers(1, 500, B)]
    arr = _states(init)
    ref = [oracle.RoundState(g, s, k) for g, s, k in init]
    for _ in range(200):
        n = [int(rng.integers(0, r.gamma + 1)) if rng.random() < 0.7 else r.gamma for r in ref]
        keep = sv.spec_round_update(arr, n, 2, 12)
        for b, r in enumerate(ref):
            k = oracle.round_update(r, n[b], 2, 12)
            assert keep[b] == k
            assert (arr[b].gamma, arr[b].seq_len, arr[b].kv_len) == (r.gamma, r.seq_len, r.kv_len)


def test_round_driver_rejects_inconsistent_state_without_changes(lib):
    arr = _states([(4, 10, 9), (4, 10, 10), (3, 5, 4)])   # sequence 1: cache and sequence disagree
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_round_update(arr, [1, 1, 1], 1, 10)
    assert e.value.code == sv.SPEC_ERR_STATE and "first bad sequence 1" in str(e.value)
    assert (arr[0].seq_len, arr[2].seq_len) == (10, 5)    # nothing was applied
    arr = _states([(4, 10, 9)])
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_round_update(arr, [5], 1, 10)             # more accepted than drafted


@pytest.mark.parametrize("gmin,gmax", [(0, 10), (5, 4), (1, 32)])
def test_round_driver_rejects_bad_bounds(lib, gmin, gmax):
    arr = _states([(4, 10, 9)])
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_round_update(arr, [1], gmin, gmax)
    assert e.value.code == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_round_update(None, None, 0, 1, 4, None, None) == sv.SPEC_ERR_INVALID_ARG
