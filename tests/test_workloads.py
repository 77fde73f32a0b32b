"""Input recipes: shapes, dtypes, determinism and the stated distributions."""
import numpy as np

import workloads as wl


def test_tiny_recipe_shapes_and_determinism():
    a = wl.make_round("tiny", r=3)
    b = wl.make_round("tiny", r=3)
    assert a.target.shape == (8, 5, 4096) and a.target.dtype == np.float32
    assert a.draft.shape == (8, 4, 4096)
    assert a.draft_tokens.shape == (8, 4) and a.draft_tokens.dtype == np.int32
    assert a.u_accept.shape == (8, 4) and a.u_resample.shape == (8,)
    assert np.array_equal(a.target, b.target) and np.array_equal(a.draft_tokens, b.draft_tokens)
    assert np.all((a.u_accept >= 0) & (a.u_accept < 1))
    assert abs(a.target.std() - 2.0) < 0.05
    assert abs((a.draft - a.target[:, :4]).std() - 0.5) < 0.02
    c = wl.make_round("tiny", r=4)
    assert not np.array_equal(a.target, c.target)


def test_uniform_stream_is_philox_seed0_in_stated_order():
    g = np.random.Generator(np.random.Philox(0))
    ua = g.random((1000, 8, 4), dtype=np.float32)
    ur = g.random((1000, 8), dtype=np.float32)
    r = wl.make_round("tiny", r=17)
    assert np.array_equal(r.u_accept, ua[17]) and np.array_equal(r.u_resample, ur[17])


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-3], dtype=np.float32)
    bits = wl.f32_to_bf16_bits(x)
    back = wl.bf16_bits_to_f32(bits)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2 ** -6 and back[3] == -2.5
    assert abs(back[4] - 1e-3) < 1e-3 * 2 ** -8


def test_zipf_profile_and_greedy_drafts():
    r = wl.make_custom(B=2, gamma=2, V=1024, dtype="bf16", profile="zipf", sigma=0.5,
                       temperature=("alternate", 0.0, 1.0))
    t = wl.bf16_bits_to_f32(r.target).astype(np.float64)
    # sorted profile follows -1.1 log(rank) up to the N(0, 0.3^2) noise
    s = np.sort(t[0, 0])[::-1]
    assert abs(np.median(s[100:900] + 1.1 * np.log(np.arange(101, 901))) ) < 0.3
    assert r.temperature[0] == 0.0 and r.temperature[1] == 1.0
    d = wl.bf16_bits_to_f32(r.draft)
    assert np.array_equal(r.draft_tokens[0], np.argmax(d[0], axis=1))


def test_lmhead_exact_sums_recipe_is_exact_in_fp32_any_order():
    """The exact-sums lm_head recipe: every logit's partial sums are exact in
    fp32, so a float32 sum in any order equals the float64 dot product."""
    B, gamma, V, H = 2, 2, 64, 1536
    W = wl.make_lmhead_W(V, H, seed=0, exact_sums=True)
    inp = wl.make_lmhead_round(0, B=B, gamma=gamma, V=V, H=H, W_bits=W, exact_sums=True)
    h = wl.bf16_bits_to_f32(inp.hidden)
    w = wl.bf16_bits_to_f32(W)
    assert np.all(np.abs(h) <= 4) and np.all(np.rint(h * 8) == h * 8)
    assert np.all(np.abs(w) <= 255 / 2048) and np.all(np.rint(w * 2048) == w * 2048)
    exact = h.astype(np.float64) @ w.astype(np.float64).T
    rng = np.random.default_rng(5)
    for r in range(h.shape[0]):
        for x in range(0, V, 7):
            prod = (h[r] * w[x]).astype(np.float32)  # exact products
            for _ in range(3):
                acc = np.float32(0)
                for t in prod[rng.permutation(H)]:
                    acc = np.float32(acc + t)
                assert float(acc) == exact[r, x]
    # the realistic recipe is not on the grid
    inp2 = wl.make_lmhead_round(0, B=B, gamma=gamma, V=V, H=H)
    assert np.any(np.rint(wl.bf16_bits_to_f32(inp2.hidden) * 8) != wl.bf16_bits_to_f32(inp2.hidden) * 8)


def test_centroid_exact_sums_recipe_is_on_the_grid_and_exact():
    """Exact-sums centroid recipe: embeddings and centroids on the 2^-11 grid
    (|k| <= 255), hidden states on the 1/8 grid (|k| <= 32); fp32 sums of the
    products in any order equal the float64 dot products."""
    m = wl.make_centroid_model(V=512, H=1536, n_clusters=16, seed=2, exact_sums=True)
    rd = wl.make_centroid_round(m, B=2, gamma=2, exact_sums=True)
    w = wl.bf16_bits_to_f32(m.W_ord)
    c = wl.bf16_bits_to_f32(m.centroids)
    h = wl.bf16_bits_to_f32(rd["hidden_draft"])
    for a in (w, c):
        assert np.all(np.abs(a) <= 255 / 2048) and np.all(np.rint(a * 2048) == a * 2048)
    assert np.all(np.abs(h) <= 4) and np.all(np.rint(h * 8) == h * 8)
    rng = np.random.default_rng(9)
    for mat in (w[::37], c):
        exact = h.astype(np.float64) @ mat.astype(np.float64).T
        for r in range(h.shape[0]):
            for x in range(mat.shape[0]):
                prod = (h[r] * mat[x]).astype(np.float32)
                acc = np.float32(0)
                for t in prod[rng.permutation(prod.size)]:
                    acc = np.float32(acc + t)
                assert float(acc) == exact[r, x]
    # cluster layout: ordered rows are grouped by cluster, ord2tok / tok2ord invert each other
    assert m.cluster_off[0] == 0 and m.cluster_off[-1] == m.V and np.all(np.diff(m.cluster_off) >= 0)
    assert np.array_equal(m.tok2ord[m.ord2tok], np.arange(m.V))
