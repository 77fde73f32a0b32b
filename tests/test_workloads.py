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
