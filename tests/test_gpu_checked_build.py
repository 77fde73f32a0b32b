"""The bounds-checked debug build (libspecverify_checked.so, built with
-DSPEC_CHECK_BOUNDS) on the small cases of the parity matrix.

In that build every checked sequence, row-slot, chunk and token index that
falls outside its extent is recorded in the status word (and the access is
skipped), so spec_verify_status returns SPEC_ERR_DEVICE_BOUNDS instead of
SPEC_OK.  compute-sanitizer is closed on this machine; this build stands in for
it on the verify path's kernels.  Each case runs in a fresh process that loads
the checked library, and the results are also held to the oracle.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import speculative_decoding_verification_54_gb300 as sv
from speculative_decoding_verification_54_gb300 import _build
sv.load(_build.build(checked=True))
import workloads as wl
import oracle
from tests.gpu_util import to_device, run_sample, run_greedy, compare, assert_tally, Tally
torch.cuda.set_device(0)
dev = torch.device("cuda:0")
t = Tally()
cases = [(5, 1, 8), (3, 31, 64), (3, 3, 3 * 8192 + 40), (2, 2, 16), (1, 4, 1024 + 8), (300, 4, 256),
         (8, 4, 4096), (4, 4, 262144)]
n = 0
for dtype in ("f32", "bf16"):
    for B, g, V in cases:
        for T in (0.9, ("alternate", 0.0, 1.3)):
            inp = wl.make_custom(B, g, V, dtype=dtype, profile="normal", target_sd=2.0, sigma=0.7,
                                 temperature=T, seed=5)
            ws = sv.make_workspace(B, g, V)
            d = to_device(inp, dev)
            tok, num, dbg, st = run_sample(sv, d, ws)
            assert st == sv.SPEC_OK, (dtype, B, g, V, T, sv.error_string(st))
            t.merge(compare(oracle.verify_sample(inp.target, inp.draft, inp.draft_tokens, inp.temperature,
                                                 inp.u_accept, inp.u_resample), tok, num, dbg))
            gt, gn, st = run_greedy(sv, d, ws)
            assert st == sv.SPEC_OK, (dtype, B, g, V, "greedy", sv.error_string(st))
            for b, r in enumerate(oracle.verify_greedy(inp.target, inp.draft_tokens)):
                assert int(gn[b]) == r.n and [int(x) for x in gt[b]] == r.tokens
            n += 1
assert_tally(t)
print("ok", n, t.checked, t.exact, t.excused)
"""


def test_checked_build_small_matrix():
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], cwd=ROOT, capture_output=True, text=True,
                       timeout=1200)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.startswith("ok"), r.stdout[-2000:]
