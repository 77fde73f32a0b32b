"""GPU (C ABI) vs fp64 oracle on the seeded workloads and the edge cases.

Every call goes through libspecverify's C entry points via the binding.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_util import (Tally, assert_tally, compare, run_greedy, run_sample,
                            to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_54_gb300 import _build
    _build.build()
    import speculative_decoding_verification_54_gb300 as m
    m.load()
    torch.cuda.set_device(0)
    return m


@pytest.fixture(scope="module")
def dev(sv):
    import torch
    return torch.device("cuda:0")


def _oracle_sample(inp, seqs=None):
    return oracle.verify_sample(inp.target, inp.draft, inp.draft_tokens, inp.temperature,
                                inp.u_accept, inp.u_resample, seqs=seqs)


def _check_sample(sv, dev, inp, ws=None, label=""):
    ws = ws if ws is not None else sv.make_workspace(inp.B, inp.gamma, inp.V)
    d = to_device(inp, dev)
    tok, num, dbg, st = run_sample(sv, d, ws)
    assert st == sv.SPEC_OK
    t = compare(_oracle_sample(inp), tok, num, dbg, label=label)
    return t, tok, num


def _check_greedy(sv, dev, inp, ws=None):
    ws = ws if ws is not None else sv.make_workspace(inp.B, inp.gamma, inp.V)
    d = to_device(inp, dev)
    tok, num, st = run_greedy(sv, d, ws)
    assert st == sv.SPEC_OK
    ref = oracle.verify_greedy(inp.target, inp.draft_tokens)
    for b, r in enumerate(ref):
        assert int(num[b]) == r.n and [int(x) for x in tok[b]] == r.tokens, (b, tok[b], r.tokens)
    return tok, num


# ---------------------------------------------------------------------------
# the five workload recipes
# ---------------------------------------------------------------------------
def test_tiny_all_rounds_sampling(sv, dev):
    ws = sv.make_workspace(8, 4, 4096)
    tally = Tally()
    ns = []
    for r in range(wl.CONFIGS["tiny"]["rounds"]):
        inp = wl.make_round("tiny", r)
        t, tok, num = _check_sample(sv, dev, inp, ws, label=f"round{r}")
        tally.merge(t)
        ns += list(num)
    assert_tally(tally)
    assert tally.checked == 8000
    # both outcomes occur: immediate rejections and fully accepted rounds (bonus)
    assert min(ns) == 0 and max(ns) == 4
    print(f"tiny sampling: {tally.exact} exact, {tally.excused} excused of {tally.checked}")


def test_tiny_all_rounds_greedy(sv, dev):
    ws = sv.make_workspace(8, 4, 4096)
    ns = []
    for r in range(wl.CONFIGS["tiny"]["rounds"]):
        inp = wl.make_round("tiny", r, temperature=0.0)
        tok, num = _check_greedy(sv, dev, inp, ws)
        ns += list(num)
        # the sampling entry point with T <= 0 is the same greedy verification
        d = to_device(inp, dev)
        tok2, num2, _, st = run_sample(sv, d, ws)
        assert st == sv.SPEC_OK and np.array_equal(tok, tok2) and np.array_equal(num, num2)
    assert min(ns) == 0 and max(ns) == 4


@pytest.mark.parametrize("sigma", [0.2, 0.5, 1.0])
def test_single_sequence_gemma_vocab(sv, dev, sigma):
    ws = sv.make_workspace(1, 4, 262144)
    tally = Tally()
    for r in range(12):
        inp = wl.make_round("single", r, sigma=sigma)
        t, _, _ = _check_sample(sv, dev, inp, ws, label=f"s{sigma}r{r}")
        tally.merge(t)
        g = wl.make_round("single", r, sigma=sigma, temperature=0.0)
        _check_greedy(sv, dev, g, ws)
    assert_tally(tally)


def test_batched_serving_full_size(sv, dev):
    """B=32, gamma=4, V=262144 bf16, T ~ U[0.5, 1.2]: the bench workload, in the
    launch configuration the bench times."""
    ws = sv.make_workspace(32, 4, 262144)
    tally = Tally()
    for r in range(2):
        inp = wl.make_round("batched", r)
        t, _, _ = _check_sample(sv, dev, inp, ws, label=f"r{r}")
        tally.merge(t)
    assert_tally(tally)


def test_long_draft_large_batch_full_size(sv, dev):
    """B=128, gamma=8, V=262144 fp32, half greedy: every sequence vs the oracle."""
    inp = wl.make_round("longdraft", 0)
    t, tok, num = _check_sample(sv, dev, inp)
    assert_tally(t)
    assert t.checked == 128
    # mixed outcomes: immediate rejections and all-accepted (bonus) rounds
    assert (num == 0).any() and (num == 8).any()


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,gamma,V", [(5, 1, 8), (3, 31, 64), (3, 3, 3 * 8192 + 40),
                                        (2, 2, 16), (1, 4, 1024 + 8), (300, 4, 256)])
def test_shapes_and_ragged_tails(sv, dev, dtype, B, gamma, V):
    for T in (0.9, ("alternate", 0.0, 1.3)):
        inp = wl.make_custom(B, gamma, V, dtype=dtype, profile="normal", target_sd=2.0,
                             sigma=0.7, temperature=T, seed=5)
        t, _, _ = _check_sample(sv, dev, inp, label=f"{dtype}{B},{gamma},{V}")
        assert_tally(t)
    g = wl.make_custom(B, gamma, V, dtype=dtype, temperature=0.0, seed=6)
    _check_greedy(sv, dev, g)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_argmax_ties_take_lowest_index(sv, dev, dtype):
    inp = wl.make_custom(6, 4, 3 * 4096 + 16, dtype=dtype, temperature=0.0, seed=8)
    rng = np.random.default_rng(8)
    vals = rng.integers(-4, 3, size=inp.target.shape).astype(np.float32)
    # plant several copies of the row maximum, across chunk boundaries
    for b in range(6):
        for j in range(5):
            pos = rng.choice(inp.V, size=5, replace=False)
            vals[b, j, pos] = 7.0
    inp.target = wl.f32_to_bf16_bits(vals) if dtype == "bf16" else vals
    # drafts: the true lowest-index argmax for some rows, a later tied index for others
    for b in range(6):
        for j in range(4):
            ties = np.flatnonzero(vals[b, j] == 7.0)
            inp.draft_tokens[b, j] = ties[0] if (b + j) % 3 else ties[-1]
    _check_greedy(sv, dev, inp)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_draft_equal_target_accepts_all_and_draws_bonus(sv, dev, dtype):
    inp = wl.make_custom(16, 5, 8192, dtype=dtype, sigma=0.0, temperature=0.8, seed=9)
    inp.draft = np.ascontiguousarray(inp.target[:, :5])
    t, tok, num = _check_sample(sv, dev, inp)
    assert_tally(t)
    assert (num == 5).all()


def test_one_hot_target_rejects_immediately(sv, dev):
    B, g, V = 4, 3, 4096
    inp = wl.make_custom(B, g, V, dtype="f32", temperature=1.0, seed=10)
    tgt = np.full((B, g + 1, V), -np.inf, dtype=np.float32)
    tgt[:, :, 77] = 0.0
    inp.target = tgt
    inp.draft_tokens[:] = 5
    inp.u_accept[:] = 0.0
    t, tok, num = _check_sample(sv, dev, inp)
    assert_tally(t)
    assert (num == 0).all() and (tok[:, 0] == 77).all()


def test_masked_minus_inf_entries(sv, dev):
    inp = wl.make_custom(8, 4, 8192, dtype="f32", temperature=1.1, seed=11)
    rng = np.random.default_rng(11)
    mask = rng.random(inp.target.shape) < 0.3
    inp.target = np.where(mask, -np.inf, inp.target).astype(np.float32)
    inp.draft = np.where(mask[:, :4], -np.inf, inp.draft).astype(np.float32)
    for b in range(8):
        for j in range(4):
            ok = np.flatnonzero(~mask[b, j])
            if not (~mask[b, j, inp.draft_tokens[b, j]]):
                inp.draft_tokens[b, j] = ok[0]
    t, _, _ = _check_sample(sv, dev, inp)
    assert_tally(t)


@pytest.mark.parametrize("T", [0.05, 5.0])
def test_extreme_temperatures(sv, dev, T):
    inp = wl.make_custom(8, 4, 16384, dtype="bf16", profile="zipf", sigma=0.5, temperature=T,
                         seed=12)
    t, _, _ = _check_sample(sv, dev, inp)
    assert_tally(t)


def test_bad_draft_token_reports_device_input_error(sv, dev):
    inp = wl.make_custom(2, 2, 1024, dtype="f32", temperature=1.0, seed=13)
    inp.draft_tokens[1, 0] = 1024  # == V
    ws = sv.make_workspace(2, 2, 1024)
    d = to_device(inp, dev)
    _, _, _, st = run_sample(sv, d, ws)
    assert st == sv.SPEC_ERR_DEVICE_INPUT
    # the status was cleared; a valid call afterwards is clean
    inp.draft_tokens[1, 0] = 3
    d = to_device(inp, dev)
    _, _, _, st = run_sample(sv, d, ws)
    assert st == sv.SPEC_OK


def test_bounded_wait_self_test_times_out_and_context_survives(sv, dev):
    ws = sv.make_workspace(4, 4, 4096)
    sv.spec_verify_selftest_timeout(ws)
    assert sv.spec_verify_status(ws) == sv.SPEC_ERR_TIMEOUT
    inp = wl.make_round("tiny", 0)
    t, _, _ = _check_sample(sv, dev, inp)
    assert_tally(t)


def test_repeat_calls_are_bitwise_deterministic(sv, dev):
    inp = wl.make_round("batched", 5)
    ws = sv.make_workspace(32, 4, 262144)
    d = to_device(inp, dev)
    a = run_sample(sv, d, ws)
    b = run_sample(sv, d, ws)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.array_equal(a[2], b[2], equal_nan=True)


_TMA_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import speculative_decoding_verification_54_gb300 as sv
import workloads as wl
from tests.gpu_util import to_device, run_sample, run_greedy
torch.cuda.set_device(0)
out = {}
for name, kw in (("bf16", dict(B=6, gamma=4, V=3 * 2048 + 24, dtype="bf16", profile="zipf",
                              temperature=("alternate", 0.0, 0.9))),
                 ("f32", dict(B=40, gamma=3, V=8192, dtype="f32", temperature=1.1))):
    inp = wl.make_custom(seed=21, **kw)
    ws = sv.make_workspace(inp.B, inp.gamma, inp.V)
    d = to_device(inp, torch.device("cuda:0"))
    tok, num, dbg, st = run_sample(sv, d, ws)
    gt, gn, st2 = run_greedy(sv, d, ws)
    assert st == 0 and st2 == 0
    out[name + "_tok"], out[name + "_num"], out[name + "_dbg"] = tok, num, dbg
    out[name + "_gtok"], out[name + "_gnum"] = gt, gn
np.savez(sys.argv[2], **out)
"""


def test_bulk_copy_load_path_matches_direct_loads(sv, tmp_path):
    """The TMA bulk-copy staging of the row reducer gives bit-identical results
    to the default direct-load path (same arithmetic, different loads)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = {}
    for path in ("ldg", "tma"):
        f = tmp_path / f"{path}.npz"
        env = dict(os.environ, SPECV_ROW_LOADS=path)
        r = subprocess.run([sys.executable, "-c", _TMA_CHILD, root, str(f)], env=env, cwd=root,
                           capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        res[path] = dict(np.load(f))
    for k in res["ldg"]:
        assert np.array_equal(res["ldg"][k], res["tma"][k], equal_nan=True), k


_CHAIN_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import speculative_decoding_verification_54_gb300 as sv
import workloads as wl
import oracle
from tests.gpu_util import to_device, run_sample, run_greedy, compare, assert_tally, Tally
torch.cuda.set_device(0)
t = Tally()
for inp in (wl.make_round("tiny", 3), wl.make_round("batched", 7),
            wl.make_custom(6, 4, 3 * 2048 + 24, dtype="bf16", profile="zipf",
                           temperature=("alternate", 0.0, 0.9), seed=21)):
    ws = sv.make_workspace(inp.B, inp.gamma, inp.V)
    d = to_device(inp, torch.device("cuda:0"))
    tok, num, dbg, st = run_sample(sv, d, ws)
    assert st == 0
    t.merge(compare(oracle.verify_sample(inp.target, inp.draft, inp.draft_tokens, inp.temperature,
                                         inp.u_accept, inp.u_resample), tok, num, dbg))
    gt, gn, st = run_greedy(sv, d, ws)
    assert st == 0
    for b, r in enumerate(oracle.verify_greedy(inp.target, inp.draft_tokens)):
        assert int(gn[b]) == r.n and [int(x) for x in gt[b]] == r.tokens
assert_tally(t)
print("ok", t.checked, t.exact, t.excused)
"""


def test_verify_chain_matches_the_oracle_in_a_fresh_process(sv):
    """The verify chain (row reducer, then tail) passes the parity checks in a
    fresh process on the tiny, batched and mixed greedy/sampled cases."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CHAIN_CHILD, root], cwd=root,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.startswith("ok")
