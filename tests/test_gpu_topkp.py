"""GPU (C ABI) vs fp64 oracle for verification with top-k / top-p truncation
of p and q (spec_verify_sample_topkp; "Gemma 4 MTP 深度解析" §5.1).

Tolerance: the logit path's (exact decisions and tokens unless a uniform lies
within 1e-6 of its boundary; probabilities within 1e-5), plus: a result may
differ where the oracle's top-p cut lies within 1e-6 (probability mass) of
top_p, since the kernel takes that decision in fp32 / two-float arithmetic.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_util import to_device

pytestmark = pytest.mark.gpu

WINDOW = 1e-6


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


def _run(sv, inp, top_k, top_p, ws=None):
    import torch
    d = to_device(inp, torch.device("cuda:0"))
    B, g1, V = d["target"].shape
    ws = ws if ws is not None else sv.make_topkp_workspace(B, g1 - 1, V)
    out = torch.full((B, g1), -7, dtype=torch.int32, device=d["target"].device)
    num = torch.full((B,), -7, dtype=torch.int32, device=d["target"].device)
    dbg = torch.zeros((B, g1, 4), dtype=torch.float32, device=d["target"].device)
    sv.spec_verify_sample_topkp(d["target"], d["draft"], d["draft_tokens"], d["temperature"], d["u_accept"],
                                d["u_resample"], top_k, top_p, out, num, ws, out_debug=dbg)
    st = sv.spec_verify_status(ws)
    return out.cpu().numpy(), num.cpu().numpy(), dbg.cpu().numpy(), st


def _compare(inp, top_k, top_p, out, num, dbg, seqs=None):
    idx = range(inp.B) if seqs is None else seqs
    ref = oracle.verify_sample_topkp(inp.target, inp.draft, inp.draft_tokens, inp.temperature, top_k, top_p,
                                     inp.u_accept, inp.u_resample, seqs=seqs)
    exact = excused = 0
    for b, r in zip(idx, ref):
        same = int(num[b]) == r.n and [int(x) for x in out[b]] == r.tokens
        near = r.margin < WINDOW or r.trunc_margin < WINDOW
        if same:
            exact += 1
        else:
            assert near, (b, int(num[b]), r.n, out[b], r.tokens, r.margin, r.trunc_margin, r.path)
            excused += 1
        if r.path != "greedy" and not near:
            for j in range(len(r.p_tok)):
                assert abs(dbg[b, j, 0] - r.p_tok[j]) <= 1e-5 and abs(dbg[b, j, 1] - r.q_tok[j]) <= 1e-5, \
                    (b, j, dbg[b, j, :2], r.p_tok[j], r.q_tok[j])
                for k, L in ((2, r.L_p[j]), (3, r.L_q[j])):
                    assert abs(dbg[b, j, k] - L) <= 1e-5 * max(1.0, abs(L)), (b, j, k, dbg[b, j, k], L)
    # the same cap as the logit path: at most 1 % of a run (at least 2) excused
    assert excused <= max(2, 0.01 * (exact + excused)), (exact, excused)
    return exact, excused


@pytest.mark.parametrize("top_k,top_p", [(64, 0.95), (1, 1.0), (5, 0.99), (1024, 1.0), (64, 0.5), (300, 0.8)])
def test_topkp_tiny_rounds(sv, top_k, top_p):
    exact = excused = 0
    for r in range(25):
        inp = wl.make_round("tiny", r)
        out, num, dbg, st = _run(sv, inp, top_k, top_p)
        assert st == sv.SPEC_OK
        e, x = _compare(inp, top_k, top_p, out, num, dbg)
        exact, excused = exact + e, excused + x
    assert excused <= 2, (exact, excused)
    print(f"top_k={top_k} top_p={top_p}: {exact} exact, {excused} excused")


def test_topkp_bf16_full_vocab_batched(sv):
    inp = wl.make_round("batched", 0)
    out, num, dbg, st = _run(sv, inp, 64, 0.95)
    assert st == sv.SPEC_OK
    e, x = _compare(inp, 64, 0.95, out, num, dbg, seqs=[0, 5, 11, 17, 23, 31])
    assert x <= 1


@pytest.mark.parametrize("top_k,top_p", [(1024, 1.0), (300, 0.8)])
def test_topkp_bf16_full_vocab_large_k(sv, top_k, top_p):
    """k at or above the number of 256-entry blocks of a 262,144-entry row
    (1,024: the block maxima bound nothing, so K comes from the sampled
    threshold) and a k below it with a deep top-p cut."""
    inp = wl.make_round("batched", 1)
    out, num, dbg, st = _run(sv, inp, top_k, top_p)
    assert st == sv.SPEC_OK
    e, x = _compare(inp, top_k, top_p, out, num, dbg, seqs=[2, 13, 29])
    assert x <= 1


def test_topkp_fp32_mixed_greedy(sv):
    inp = wl.make_custom(16, 8, 262144, "f32", "zipf", sigma=("uniform", 0.1, 1.5),
                         temperature=("alternate", 0.0, 1.0), seed=3)
    out, num, dbg, st = _run(sv, inp, 64, 0.9)
    assert st == sv.SPEC_OK
    e, x = _compare(inp, 64, 0.9, out, num, dbg, seqs=[0, 1, 6, 9, 14, 15])
    assert x <= 1


def test_topkp_ties_at_the_boundary(sv):
    """Logits quantised to a coarse grid: many ties at the top_k-th value,
    kept as a group on both sides."""
    inp = wl.make_custom(8, 4, 8192, "f32", "normal", target_sd=2.0, sigma=0.5, temperature=1.0, seed=9)
    inp.target[:] = np.round(inp.target * 2) / 2
    inp.draft[:] = np.round(inp.draft * 2) / 2
    for k, tp in ((16, 1.0), (64, 0.9)):
        out, num, dbg, st = _run(sv, inp, k, tp)
        assert st == sv.SPEC_OK
        _compare(inp, k, tp, out, num, dbg)


def test_topkp_list_overflow_is_reported(sv):
    inp = wl.make_custom(2, 2, 8192, "f32", "normal", seed=4)
    inp.target[:] = 0.0   # every entry ties with the maximum: K holds all 8192
    out, num, dbg, st = _run(sv, inp, 8, 1.0)
    assert st == sv.SPEC_ERR_UNSUPPORTED
