"""GPU (C ABI) vs fp64 oracle for several draft candidates per sequence
(spec_verify_greedy_multi; "Accelerating Gemma 4…" §6, item 2 多候选草稿):
bit-exact kept candidate, accepted count and tokens."""
import numpy as np
import pytest

import oracle
import workloads as wl

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


def _run(sv, target, toks):
    import torch
    dev = torch.device("cuda:0")
    B, n, g1, V = target.shape
    if target.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(target).view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(target)).to(dev)
    d = torch.from_numpy(np.ascontiguousarray(toks)).to(dev)
    out = torch.full((B, g1), -7, dtype=torch.int32, device=dev)
    num = torch.full((B,), -7, dtype=torch.int32, device=dev)
    ch = torch.full((B,), -7, dtype=torch.int32, device=dev)
    ws = sv.make_workspace(B * n, g1 - 1, V)
    sv.spec_verify_greedy_multi(t, d, out, num, ws, out_choice=ch)
    assert sv.spec_verify_status(ws) == sv.SPEC_OK
    return out.cpu().numpy(), num.cpu().numpy(), ch.cpu().numpy()


def _check(target, toks, out, num, ch):
    ref = oracle.verify_greedy_multi(target, toks)
    for b, (r, c) in enumerate(ref):
        assert int(ch[b]) == c and int(num[b]) == r.n and [int(x) for x in out[b]] == r.tokens, \
            (b, int(ch[b]), c, int(num[b]), r.n, out[b], r.tokens)
    return [r.n for r, _ in ref]


def test_multi_small_fp32_varied_lengths(sv):
    """Candidates accept 0..gamma drafts: drafts are argmax-chain prefixes of
    chosen lengths followed by a wrong token; some sequences have ties."""
    rng = np.random.default_rng(3)
    B, n, g, V = 6, 4, 5, 4096 + 8
    tgt = rng.normal(0, 2, (B, n, g + 1, V)).astype(np.float32)
    toks = np.zeros((B, n, g), np.int32)
    for b in range(B):
        for c in range(n):
            k = int(rng.integers(0, g + 1)) if b % 2 else (2 if c in (1, 3) else 1)  # even b: a tie at 2
            for j in range(g):
                a = int(np.argmax(tgt[b, c, j]))
                toks[b, c, j] = a if j < k else (a + 1 + int(rng.integers(0, V - 1))) % V
    out, num, ch = _run(sv, tgt, toks)
    ns = _check(tgt, toks, out, num, ch)
    assert ch[0] == 1 and ch[2] == 1  # ties at n = 2 keep the lower index
    assert len(set(ns)) > 1


def test_multi_bf16_full_vocab(sv):
    tgt, toks = wl.make_multi(8, 4, gamma=4, V=262144, dtype="bf16", profile="zipf", seed=5)
    out, num, ch = _run(sv, tgt, toks)
    _check(tgt, toks, out, num, ch)


def test_multi_many_candidates_and_one(sv):
    tgt, toks = wl.make_multi(3, 40, gamma=3, V=2048, seed=7)  # more candidates than lanes
    out, num, ch = _run(sv, tgt, toks)
    _check(tgt, toks, out, num, ch)
    tgt1, toks1 = wl.make_multi(5, 1, gamma=4, V=4096, seed=8)
    out, num, ch = _run(sv, tgt1, toks1)
    _check(tgt1, toks1, out, num, ch)
    assert (ch == 0).all()
