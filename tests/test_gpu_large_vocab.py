"""GPU (C ABI) vs the fp64 oracle at the largest vocabularies.

V = 2^23 + 8 gives 4,097 chunks of 2,048 bf16 entries per row: one more than
the tail stages in shared memory for the draw (4,096 chunk masses), so the
draw scans the masses from memory, and the last chunk holds 8 entries.
V = 2^26 is the largest vocabulary the C ABI accepts (SPEC_MAX_VOCAB), with
32,768 chunks per row.  Same tolerance as the other parity tests.
"""
import pytest

import workloads as wl
from tests.gpu_util import assert_tally
from tests.test_gpu_parity import _check_greedy, _check_sample, dev, sv  # noqa: F401  (fixtures)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,gamma,V,T", [(1, 3, (1 << 23) + 8, 0.9), (1, 1, 1 << 26, 1.0)])
def test_largest_vocabularies(sv, dev, B, gamma, V, T):
    inp = wl.make_custom(B, gamma, V, dtype="bf16", profile="normal", target_sd=2.0, sigma=0.5,
                         temperature=T, seed=11)
    t, _, _ = _check_sample(sv, dev, inp, label=f"V{V}")
    assert_tally(t)
    g = wl.make_custom(B, gamma, V, dtype="bf16", profile="normal", temperature=0.0, seed=12)
    _check_greedy(sv, dev, g)
