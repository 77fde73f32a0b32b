"""GPU (C ABI) vs fp64 oracle for the centroid-masked sparse draft head and
the verification against its sparse rows ("Gemma 4 MTP 深度解析" §3.4
Centroids Masking; "Gemma 4 - Drafter 解析", 高效 Embedder).

Head: on the exact-sums recipe every dot product is exact in fp32, so cluster
selection, candidate sets and logits must equal the oracle bit for bit.
Sparse verification: the logit path's tolerance (exact decisions and tokens
unless a uniform lies within 1e-6 of its boundary; probabilities within
1e-5); candidates enter both sides as the same float32 values.
"""
import numpy as np
import pytest

import oracle
import workloads as wl

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


def _bf16(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def _i32(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def _run_head(sv, model, hidden_bits, top_k, max_cand=8192):
    import torch
    dev = torch.device("cuda:0")
    R = hidden_bits.shape[0]
    out_tok = torch.full((R, max_cand), -5, dtype=torch.int32, device=dev)
    out_log = torch.full((R, max_cand), float("nan"), dtype=torch.float32, device=dev)
    cnt = torch.full((R,), -5, dtype=torch.int32, device=dev)
    ws = sv.make_centroid_head_workspace(R, model.n_clusters, top_k, device=dev)
    sv.spec_centroid_head(_bf16(hidden_bits, dev), _bf16(model.centroids, dev), _bf16(model.W_ord, dev),
                          _i32(model.cluster_off, dev), _i32(model.ord2tok, dev), top_k, out_tok, out_log, cnt, ws)
    st = sv.spec_verify_status(ws)
    return out_tok.cpu().numpy(), out_log.cpu().numpy(), cnt.cpu().numpy(), st


def test_head_exact_small(sv):
    m = wl.make_centroid_model(V=16384, H=256, n_clusters=128, seed=4, exact_sums=True, mu_sd=0.12, eps_sd=0.005)
    rd = wl.make_centroid_round(m, B=4, gamma=3, exact_sums=True, draft_sd=0.05)
    for top_k in (1, 8, 48):  # 48 of 128 clusters: about 6,100 candidates
        tok, lg, cnt, st = _run_head(sv, m, rd["hidden_draft"], top_k)
        assert st == sv.SPEC_OK
        ref = oracle.centroid_head(rd["hidden_draft"], m.centroids, m.W_ord, m.cluster_off, m.ord2tok, top_k)
        for r, (t_ref, l_ref) in enumerate(ref):
            assert cnt[r] == len(t_ref), (top_k, r)
            assert np.array_equal(tok[r, :cnt[r]], t_ref)
            assert np.array_equal(lg[r, :cnt[r]].astype(np.float64), l_ref)  # exact recipe: bitwise


@pytest.mark.parametrize("B,gamma,n_clusters,H,top_k", [
    (12, 3, 200, 512, 24),   # R = 36: one row chunk of 48, a ragged last 128-cluster tile
    (100, 3, 256, 256, 16),  # R = 300: two row chunks (256 + 44), four K steps
])
def test_head_exact_tensor_core_scores(sv, B, gamma, n_clusters, H, top_k):
    """More than 16 hidden rows: the cluster scores come from the tcgen05
    GEMM with K split over several CTAs; on the exact-sums recipe the
    selection, the candidates and their logits equal the oracle bitwise."""
    m = wl.make_centroid_model(V=16384, H=H, n_clusters=n_clusters, seed=9, exact_sums=True, mu_sd=0.12,
                               eps_sd=0.005)
    rd = wl.make_centroid_round(m, B=B, gamma=gamma, exact_sums=True, draft_sd=0.05)
    assert rd["hidden_draft"].shape[0] == B * gamma > 16
    tok, lg, cnt, st = _run_head(sv, m, rd["hidden_draft"], top_k)
    assert st == sv.SPEC_OK
    ref = oracle.centroid_head(rd["hidden_draft"], m.centroids, m.W_ord, m.cluster_off, m.ord2tok, top_k)
    for r, (t_ref, l_ref) in enumerate(ref):
        assert cnt[r] == len(t_ref), r
        assert np.array_equal(tok[r, :cnt[r]], t_ref), r
        assert np.array_equal(lg[r, :cnt[r]].astype(np.float64), l_ref), r


def test_head_exact_past_the_bitmap_vocabulary(sv):
    """Above 262,144 tokens the candidates are ordered by the sort kernel (a
    bitonic sort) instead of the selection kernel's ranks; same bar: bitwise."""
    m = wl.make_centroid_model(V=262144 + 4096, H=256, n_clusters=64, seed=8, exact_sums=True, mu_sd=0.12,
                               eps_sd=0.005)
    rd = wl.make_centroid_round(m, B=2, gamma=1, exact_sums=True, draft_sd=0.05)
    tok, lg, cnt, st = _run_head(sv, m, rd["hidden_draft"], 1)  # one cluster: about 4,160 candidates
    assert st == sv.SPEC_OK
    ref = oracle.centroid_head(rd["hidden_draft"], m.centroids, m.W_ord, m.cluster_off, m.ord2tok, 1)
    for r, (t_ref, l_ref) in enumerate(ref):
        assert cnt[r] == len(t_ref)
        assert np.array_equal(tok[r, :cnt[r]], t_ref)
        assert np.array_equal(lg[r, :cnt[r]].astype(np.float64), l_ref)


def test_head_all_clusters_is_every_token(sv):
    m = wl.make_centroid_model(V=4096, H=512, n_clusters=64, seed=5, exact_sums=True)
    rd = wl.make_centroid_round(m, B=2, gamma=2, exact_sums=True)
    tok, lg, cnt, st = _run_head(sv, m, rd["hidden_draft"], 64)
    assert st == sv.SPEC_OK
    dense = oracle.lmhead_logits(rd["hidden_draft"], m.W_ord[m.tok2ord])
    for r in range(tok.shape[0]):
        assert cnt[r] == 4096 and np.array_equal(tok[r, :4096], np.arange(4096))
        assert np.array_equal(lg[r, :4096].astype(np.float64), dense[r])


def test_head_ties_keep_the_lowest_cluster(sv):
    m = wl.make_centroid_model(V=4096, H=256, n_clusters=64, seed=6, exact_sums=True)
    m.centroids[17] = m.centroids[3]  # clusters 3 and 17 always tie
    m.centroids[40] = m.centroids[3]
    rd = wl.make_centroid_round(m, B=3, gamma=2, exact_sums=True)
    tok, lg, cnt, st = _run_head(sv, m, rd["hidden_draft"], 5)
    ref = oracle.centroid_head(rd["hidden_draft"], m.centroids, m.W_ord, m.cluster_off, m.ord2tok, 5)
    for r, (t_ref, _) in enumerate(ref):
        assert np.array_equal(tok[r, :cnt[r]], t_ref)


def test_head_overflow_is_reported(sv):
    m = wl.make_centroid_model(V=4096, H=256, n_clusters=16, seed=7)
    rd = wl.make_centroid_round(m, B=1, gamma=2)
    tok, lg, cnt, st = _run_head(sv, m, rd["hidden_draft"], 8, max_cand=256)  # 8 clusters hold ~2048 tokens
    assert st == sv.SPEC_ERR_UNSUPPORTED
    assert np.all(cnt == 256)


def test_head_full_size_exact(sv):
    """V=262,144, H=1,536, 2,048 clusters, top 32 (the pages' shape), exact-sums
    embeddings drawn with torch on the GPU, checked on every row."""
    import torch
    dev = torch.device("cuda:0")
    V, H, Nc, top_k, R = 262144, 1536, 2048, 32, 8
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    cl = torch.randint(0, Nc, (V,), generator=g, device=dev)
    key = cl.to(torch.int64) * V + torch.arange(V, device=dev)
    ord2tok = torch.argsort(key).to(torch.int32)
    counts = torch.bincount(cl, minlength=Nc)
    off = torch.zeros(Nc + 1, dtype=torch.int32, device=dev)
    off[1:] = torch.cumsum(counts, 0).to(torch.int32)
    mu = 0.05 * torch.randn(Nc, H, generator=g, device=dev)
    w = mu[cl[ord2tok.long()]] + 0.004 * torch.randn(V, H, generator=g, device=dev)
    w = (torch.clamp(torch.round(w * 2048), -255, 255) / 2048).to(torch.bfloat16)
    sums = torch.zeros(Nc, H, device=dev).index_add_(0, cl[ord2tok.long()], w.float())
    cen = torch.where(counts[:, None] > 0, sums / counts.clamp(min=1)[:, None], mu)
    cen = (torch.clamp(torch.round(cen * 2048), -255, 255) / 2048).to(torch.bfloat16)
    hid = (torch.clamp(torch.round(torch.randn(R, H, generator=g, device=dev) * 8), -32, 32) / 8).to(torch.bfloat16)
    del sums, mu
    max_cand = 8192
    out_tok = torch.full((R, max_cand), -5, dtype=torch.int32, device=dev)
    out_log = torch.zeros((R, max_cand), dtype=torch.float32, device=dev)
    cnt = torch.zeros((R,), dtype=torch.int32, device=dev)
    ws = sv.make_centroid_head_workspace(R, Nc, top_k, device=dev)
    sv.spec_centroid_head(hid, cen, w, off, ord2tok, top_k, out_tok, out_log, cnt, ws)
    assert sv.spec_verify_status(ws) == sv.SPEC_OK
    to_bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.centroid_head(to_bits(hid), to_bits(cen), to_bits(w), off.cpu().numpy(), ord2tok.cpu().numpy(),
                               top_k)
    tok, lg, cnt = out_tok.cpu().numpy(), out_log.cpu().numpy(), cnt.cpu().numpy()
    for r, (t_ref, l_ref) in enumerate(ref):
        assert cnt[r] == len(t_ref) and 3000 < cnt[r] < 5200
        assert np.array_equal(tok[r, :cnt[r]], t_ref)
        assert np.array_equal(lg[r, :cnt[r]].astype(np.float64), l_ref)


# ---------------------------------------------------------------------------
# sparse verification
# ---------------------------------------------------------------------------
def _cand_arrays(cand, stride):
    n = len(cand)
    tok = np.zeros((n, stride), np.int32)
    lg = np.zeros((n, stride), np.float32)
    cnt = np.zeros(n, np.int32)
    for i, (t, l) in enumerate(cand):
        k = min(len(t), stride)
        tok[i, :k], lg[i, :k], cnt[i] = t[:k], np.asarray(l[:k], np.float32), k
    return tok, lg, cnt


def _run_sparse(sv, target_bits, cand, draft_tokens, temperature, ua, ur, stride=8192):
    import torch
    dev = torch.device("cuda:0")
    B, g1, V = target_bits.shape
    tok, lg, cnt = _cand_arrays(cand, stride)
    out = torch.full((B, g1), -7, dtype=torch.int32, device=dev)
    num = torch.full((B,), -7, dtype=torch.int32, device=dev)
    dbg = torch.zeros((B, g1, 4), dtype=torch.float32, device=dev)
    ws = sv.make_sparse_workspace(B, g1 - 1, V, device=dev)
    tgt = _bf16(target_bits, dev) if target_bits.dtype == np.uint16 else torch.from_numpy(target_bits).to(dev)
    sv.spec_verify_sample_sparse(tgt, _i32(tok, dev), torch.from_numpy(lg).to(dev), _i32(cnt, dev),
                                 _i32(draft_tokens, dev), torch.from_numpy(np.asarray(temperature, np.float32)).to(dev),
                                 torch.from_numpy(np.ascontiguousarray(ua)).to(dev),
                                 torch.from_numpy(np.ascontiguousarray(ur)).to(dev), out, num, ws, out_debug=dbg)
    st = sv.spec_verify_status(ws)
    return out.cpu().numpy(), num.cpu().numpy(), dbg.cpu().numpy(), st


def _compare_sparse(target, cand, d, temp, ua, ur, out, num, dbg, gamma, seqs=None):
    B = len(d)
    idx = range(B) if seqs is None else seqs
    c32 = [(t, np.asarray(l, np.float32).astype(np.float64)) for (t, l) in cand]
    per_seq = [[c32[b * gamma + j] for j in range(gamma)] for b in range(B)]
    ref = oracle.verify_sample_sparse(target, per_seq, d, temp, ua, ur, seqs=list(idx))
    exact = excused = 0
    for b, r in zip(idx, ref):
        same = int(num[b]) == r.n and [int(x) for x in out[b]] == r.tokens
        if same:
            exact += 1
        else:
            assert r.margin < WINDOW, (b, int(num[b]), r.n, out[b], r.tokens, r.margin, r.path)
            excused += 1
        if r.path != "greedy" and r.margin >= WINDOW:
            for j in range(len(r.p_tok)):
                assert abs(dbg[b, j, 0] - r.p_tok[j]) <= 1e-5 and abs(dbg[b, j, 1] - r.q_tok[j]) <= 1e-5
                for k, L in ((2, r.L_p[j]), (3, r.L_q[j])):
                    if np.isinf(L):
                        assert dbg[b, j, k] == L, (b, j, k, dbg[b, j, k], L)  # a row without candidates
                    else:
                        assert abs(dbg[b, j, k] - L) <= 1e-5 * max(1.0, abs(L)), (b, j, k, dbg[b, j, k], L)
    return exact, excused


def _sparse_round(seed, B=8, gamma=3, V=16384, H=256, Nc=128, top_k=8, T=0.7, r=0):
    m = wl.make_centroid_model(V=V, H=H, n_clusters=Nc, seed=seed, mu_sd=0.12, eps_sd=0.005)
    rd = wl.make_centroid_round(m, B=B, gamma=gamma, r=r, draft_sd=0.05, temperature=T)
    cand = oracle.centroid_head(rd["hidden_draft"], m.centroids, m.W_ord, m.cluster_off, m.ord2tok, top_k)
    cand = [(t, np.asarray(l, np.float32)) for (t, l) in cand]
    d = wl.sample_sparse_drafts(cand, rd["temperature"], gamma, r=r)
    return rd, cand, d


@pytest.mark.parametrize("T", [0.7, 1.0, ("alternate", 0.0, 0.8)])
def test_sparse_verify_small_rounds(sv, T):
    exact = excused = 0
    paths = set()
    for r in range(6):
        temp = T if not isinstance(T, tuple) else np.where(np.arange(8) % 2 == 0, 0.0, 0.8)
        rd, cand, d = _sparse_round(seed=20 + r, T=temp, r=r)
        out, num, dbg, st = _run_sparse(sv, rd["target"], cand, d, rd["temperature"], rd["u_accept"], rd["u_resample"])
        assert st == sv.SPEC_OK
        e, x = _compare_sparse(rd["target"], cand, d, rd["temperature"], rd["u_accept"], rd["u_resample"],
                               out, num, dbg, 3)
        exact, excused = exact + e, excused + x
        paths |= {int(n) for n in num}
    assert excused <= 1
    assert len(paths) >= 2  # both rejections and full acceptances occur


def test_sparse_verify_edge_cases(sv):
    """Empty candidate rows (q = 0: every draft accepted), a single candidate,
    drafts that are not candidates, gamma = 1."""
    rd, cand, d = _sparse_round(seed=31, B=6, gamma=3)
    cand = list(cand)
    cand[0] = (np.zeros(0, np.int64), np.zeros(0, np.float32))  # seq 0, row 0: no candidates
    cand[1] = (cand[1][0][:1], cand[1][1][:1])                    # seq 0, row 1: one candidate
    d = d.copy()
    d[1, 0] = int(np.setdiff1d(np.arange(16384), cand[3][0])[5])  # seq 1: draft outside its candidates
    out, num, dbg, st = _run_sparse(sv, rd["target"], cand, d, rd["temperature"], rd["u_accept"], rd["u_resample"])
    assert st == sv.SPEC_OK
    _compare_sparse(rd["target"], cand, d, rd["temperature"], rd["u_accept"], rd["u_resample"], out, num, dbg, 3)
    rd1, cand1, d1 = _sparse_round(seed=32, B=5, gamma=1)
    out, num, dbg, st = _run_sparse(sv, rd1["target"], cand1, d1, rd1["temperature"], rd1["u_accept"],
                                    rd1["u_resample"])
    _compare_sparse(rd1["target"], cand1, d1, rd1["temperature"], rd1["u_accept"], rd1["u_resample"], out, num, dbg, 1)


def test_sparse_verify_full_vocab_batched(sv):
    """B=32, gamma=4, V=262,144 bf16 targets (Zipf recipe) with 4,096 sorted
    random candidates per draft row whose logits follow the target's; checked
    on sampled sequences; run twice for determinism."""
    inp = wl.make_round("batched", 0)
    rng = np.random.default_rng(5)
    cand = []
    tgt = wl.bf16_bits_to_f32(inp.target)
    for b in range(inp.B):
        for j in range(inp.gamma):
            t = np.sort(rng.choice(inp.V, 4096, replace=False))
            t[rng.integers(0, 4096)] = np.argmax(tgt[b, j])  # keep the mode in the list
            t = np.unique(t)
            cand.append((t, (tgt[b, j, t] + rng.normal(0, 0.3, t.size)).astype(np.float32)))
    d = wl.sample_sparse_drafts(cand, inp.temperature, inp.gamma, r=3)
    out, num, dbg, st = _run_sparse(sv, inp.target, cand, d, inp.temperature, inp.u_accept, inp.u_resample)
    assert st == sv.SPEC_OK
    out2, num2, _, _ = _run_sparse(sv, inp.target, cand, d, inp.temperature, inp.u_accept, inp.u_resample)
    assert np.array_equal(out, out2) and np.array_equal(num, num2)
    e, x = _compare_sparse(inp.target, cand, d, inp.temperature, inp.u_accept, inp.u_resample, out, num, dbg,
                           inp.gamma, seqs=[0, 7, 13, 21, 30])
    assert x <= 1
