"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

None of these re-types an oracle formula.  They use printed values from the
pages (tests/golden/), closed forms, exhaustive enumeration of a toy model,
brute-force loops and independent library routines.  The mutation tests at
the end plant plausible mistakes in the oracle (on the CPU) and show that a
pin catches each one.
"""
import json
import math
import os
from functools import lru_cache

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import spec_oracle as so

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# input widening, softmax, argmax
# ---------------------------------------------------------------------------
def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F7F, 0x0001, 0xFF80],
                    dtype=np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 0.0, -0.0, (2 - 2 ** -7) * 2.0 ** 127,
            2.0 ** -133, -math.inf]
    got = so.bf16_bits_to_f64(bits)
    for g, w in zip(got, want):
        assert g == w


@pytest.mark.parametrize("T", [0.5, 0.7, 1.0, 1.2, 3.0])
def test_log_normaliser_matches_scipy_logsumexp(T):
    rng = np.random.default_rng(11)
    for V in (8, 4096, 262144):
        x = rng.normal(0, 4, V)
        L = so.row_log_normaliser(x, T)
        assert abs(L - scipy.special.logsumexp(x / T)) <= 1e-12 * max(1.0, abs(L))
        p = so.row_probs(x, T)
        assert abs(math.fsum(p) - 1.0) < 1e-12
        # softmax ratio identity: p_a / p_b = exp((x_a - x_b)/T)
        a, b = 3, 5
        assert abs(p[a] / p[b] - math.exp((x[a] - x[b]) / T)) < 1e-9 * p[a] / p[b]


def test_log_normaliser_with_masked_entries():
    x = np.array([0.0, -np.inf, math.log(3.0), -np.inf])
    assert abs(so.row_log_normaliser(x, 1.0) - math.log(4.0)) < 1e-15
    assert so.row_probs(x, 1.0)[1] == 0.0


def test_argmax_lowest_index_on_ties_matches_numpy():
    rng = np.random.default_rng(5)
    for _ in range(200):
        x = rng.integers(-3, 4, size=rng.integers(1, 64)).astype(np.float64)
        assert so.row_argmax(x) == int(np.argmax(x))  # numpy returns the first max


# ---------------------------------------------------------------------------
# the worked example of the book chapter (golden fixture)
# ---------------------------------------------------------------------------
def _one_hot_rows(choices, V, hi=5.0):
    rows = np.zeros((len(choices), V))
    for j, c in enumerate(choices):
        rows[j, c] = hi
    return rows


def worked_example_failures(verify=None):
    verify = verify or so.verify_greedy_seq
    g = _golden("book_ch8_worked_example.json")
    vocab = {t: i for i, t in enumerate(g["vocab"])}
    tn = g["target_next"]
    target_next = [vocab[tn[k]] for k in ("row0_after_context", "row1_after_我",
                                           "row2_after_我们", "row3_after_我们去",
                                           "row4_after_我们去园")]
    rows = _one_hot_rows(target_next, len(vocab))
    bad = 0
    for case in ("case_mismatch", "case_all_correct"):
        c = g[case]
        drafts = [vocab[t] for t in c["drafts"]]
        res = verify(rows, drafts)
        want = [vocab[t] for t in c["expected_output"]]
        ok = (res.n == c["expected_accepted"] and res.tokens[:res.n + 1] == want
              and all(t == -1 for t in res.tokens[res.n + 1:]))
        bad += not ok
    return bad


def test_worked_example_book_ch8():
    assert worked_example_failures() == 0


# ---------------------------------------------------------------------------
# a toy prefix-keyed language model (test-only; not oracle code)
# ---------------------------------------------------------------------------
def _toy_logits(prefix, salt, V, sd):
    ss = np.random.SeedSequence([salt, V, len(prefix), *prefix])
    return np.random.default_rng(ss).normal(0.0, sd, V)


class ToyLM:
    """p(.|prefix) and q(.|prefix) over V tokens, fixed by hashing the prefix."""

    def __init__(self, V, salt=0, sd=1.5, draft_noise=0.8):
        self.V, self.salt, self.sd, self.dn = V, salt, sd, draft_noise

    def target_logits(self, prefix):
        return _toy_logits(tuple(prefix), self.salt, self.V, self.sd)

    def draft_logits(self, prefix):
        return self.target_logits(prefix) + self.dn * _toy_logits(tuple(prefix), self.salt + 1000, self.V, 1.0)


def _greedy_chain(lm, prompt, n):
    pre, out = list(prompt), []
    for _ in range(n):
        t = int(np.argmax(lm.target_logits(pre)))
        out.append(t)
        pre.append(t)
    return out


def _spec_greedy(lm, prompt, n, gamma, verify=None):
    verify = verify or so.verify_greedy_seq
    pre, out = list(prompt), []
    while len(out) < n:
        drafts, cur = [], list(pre)
        for _ in range(gamma):
            d = int(np.argmax(lm.draft_logits(cur)))
            drafts.append(d)
            cur.append(d)
        rows = np.stack([lm.target_logits(pre + drafts[:j]) for j in range(gamma + 1)])
        res = verify(rows, drafts)
        emitted = res.tokens[:res.n + 1]
        assert len(emitted) >= 1 and -1 not in emitted
        out += emitted
        pre += emitted
    return out[:n]


def greedy_chain_mismatches(verify=None):
    bad = 0
    for salt in range(6):
        for gamma in (1, 2, 4, 7):
            lm = ToyLM(V=8, salt=salt)
            bad += _spec_greedy(lm, [salt % 8], 24, gamma, verify) != _greedy_chain(lm, [salt % 8], 24)
    return bad


def test_greedy_speculation_equals_plain_argmax_chain():
    """Greedy speculative output is bit-identical to the target's own greedy
    output ("Gemma 4 MTP 深度解析" §2.2; "自投机解码…" §3.1)."""
    assert greedy_chain_mismatches() == 0


# ---------------------------------------------------------------------------
# several draft candidates ("Accelerating Gemma 4…" §6, item 2 多候选草稿)
# ---------------------------------------------------------------------------
def _cand_drafts(lm, pre, gamma, c):
    """Greedy drafts of candidate c: its own noisy draft model (salt per c)."""
    cur, drafts = list(pre), []
    for _ in range(gamma):
        lq = lm.target_logits(cur) + lm.dn * _toy_logits(tuple(cur), lm.salt + 1000 + 17 * c, lm.V, 1.0)
        d = int(np.argmax(lq))
        drafts.append(d)
        cur.append(d)
    return drafts


def multi_candidate_failures(verify_multi=None):
    """Decode with n candidates per round; the output must be the plain argmax
    chain, and each round must keep as many drafts as the best candidate's
    common prefix with that chain."""
    verify_multi = verify_multi or so.verify_greedy_multi
    bad = 0
    for salt in range(4):
        for gamma in (2, 4):
            for n_cand in (2, 3, 5):
                lm = ToyLM(V=8, salt=salt, draft_noise=1.2)
                chain = _greedy_chain(lm, [salt % 8], 40)
                pre, out = [salt % 8], []
                while len(out) < 24:
                    cands = [_cand_drafts(lm, pre, gamma, c) for c in range(n_cand)]
                    target = np.stack([np.stack([lm.target_logits(pre + d[:j]) for j in range(gamma + 1)])
                                       for d in cands])[None]
                    res, choice = verify_multi(target, np.array(cands)[None])[0]
                    ref = chain[len(out):len(out) + gamma + 1]
                    best = max(next((j for j in range(gamma) if d[j] != ref[j]), gamma) for d in cands)
                    emitted = res.tokens[:res.n + 1]
                    bad += (res.n != best) + (emitted != ref[:len(emitted)]) + (cands[choice][:res.n] != ref[:res.n])
                    out += emitted
                    pre += emitted
    return bad


def test_multi_candidate_keeps_the_longest_and_matches_the_argmax_chain():
    assert multi_candidate_failures() == 0


def test_multi_candidate_ties_and_single_candidate():
    rng = np.random.default_rng(41)
    g, V = 3, 16
    rows = rng.normal(0, 2, (g + 1, V))
    chain = [int(np.argmax(rows[j])) for j in range(g)]
    bad_draft = [(chain[0] + 1) % V] + chain[1:]
    # two equally good candidates: the lower index is kept
    t = np.stack([rows, rows])[None]
    res, choice = so.verify_greedy_multi(t, np.array([[chain, chain]]))[0]
    assert choice == 0 and res.n == g
    # the strictly better candidate wins wherever it sits
    res, choice = so.verify_greedy_multi(t, np.array([[bad_draft, chain]]))[0]
    assert choice == 1 and res.n == g
    # one candidate: plain greedy verification
    res, choice = so.verify_greedy_multi(rows[None, None], np.array([[bad_draft]]))[0]
    assert choice == 0 and res.tokens == so.verify_greedy_seq(rows, bad_draft).tokens


# ---------------------------------------------------------------------------
# exhaustive enumeration: the output marginal equals the target's own
# autoregressive distribution ("Gemma 4 MTP 深度解析" §2.2; "第 8 章…" 为什么输出不会变)
# ---------------------------------------------------------------------------
def _round_distribution(lm, prefix, gamma, T, mod):
    """Exact distribution of the tokens one verify round emits from ``prefix``.
    Uses the oracle's acceptance probability and residual weights; the drafts
    are drawn from q (enumerated)."""
    V = lm.V
    P = lambda pre: mod.row_probs(lm.target_logits(pre), T)
    Q = lambda pre: mod.row_probs(lm.draft_logits(pre), T)
    dist = {}

    def add(seq, w):
        if w > 0:
            dist[seq] = dist.get(seq, 0.0) + w

    def walk(pre, drafts, weight):
        j = len(drafts)
        p, = (P(pre + drafts),)
        if j == gamma:
            for t in range(V):
                add(tuple(drafts) + (t,), weight * p[t])
            return
        q = Q(pre + drafts)
        r = mod.residual_weights(p, q)
        z = r.sum()
        for d in range(V):
            if q[d] == 0:
                continue
            a = mod.acceptance_probability(p, q, d)
            if a < 1 and z > 0:
                for t in range(V):
                    add(tuple(drafts) + (t,), weight * q[d] * (1 - a) * r[t] / z)
            walk(pre, drafts + [d], weight * q[d] * a)

    walk(list(prefix), [], 1.0)
    return dist


def lossless_enumeration_error(mod=so, V=8, gamma=2, T=1.0, k=3, salt=3):
    lm = ToyLM(V=V, salt=salt, sd=1.2, draft_noise=1.0)

    @lru_cache(maxsize=None)
    def first_k(prefix, kk):
        out = {}
        for seq, w in _round_distribution(lm, list(prefix), gamma, T, mod).items():
            if len(seq) >= kk:
                out[seq[:kk]] = out.get(seq[:kk], 0.0) + w
            else:
                for rest, w2 in first_k(prefix + seq, kk - len(seq)).items():
                    out[seq + rest] = out.get(seq + rest, 0.0) + w * w2
        return out

    spec = first_k((1,), k)
    err = 0.0
    for t1 in range(V):
        p1 = scipy.special.softmax(lm.target_logits([1]) / T)[t1]
        for t2 in range(V):
            p2 = scipy.special.softmax(lm.target_logits([1, t1]) / T)[t2]
            for t3 in range(V):
                p3 = scipy.special.softmax(lm.target_logits([1, t1, t2]) / T)[t3]
                err = max(err, abs(spec.get((t1, t2, t3), 0.0) - p1 * p2 * p3))
    return err


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_lossless_marginal_exact_enumeration_V8_gamma2(T):
    assert lossless_enumeration_error(T=T) < 1e-12


# ---------------------------------------------------------------------------
# expected tokens per round (closed form printed on the pages)
# ---------------------------------------------------------------------------
def _two_token_toy(gamma):
    """V=2: q = (1, 0), p = (0.8, 0.2) at every position: alpha = 0.8 exactly."""
    tgt = np.tile(np.log([0.8, 0.2]), (gamma + 1, 1))
    dft = np.tile(np.array([0.0, -np.inf]), (gamma, 1))
    return tgt, dft


def test_closed_form_expected_tokens_printed_value():
    g = _golden("closed_forms.json")["expected_tokens"]
    E = oracle.expected_tokens_per_round(g["alpha"], g["gamma"])
    assert round(E, g["printed_decimals"]) == g["printed_value"]
    # the closed form equals the term-by-term sum 1 + alpha + ... + alpha^gamma
    assert abs(E - math.fsum(g["alpha"] ** k for k in range(g["gamma"] + 1))) < 1e-15


def test_tokens_per_round_exact_matches_closed_form():
    """Exact distribution of the emitted count from the oracle's acceptance
    probability, against (1 - a^(g+1)) / (1 - a)."""
    for gamma in (1, 4, 8):
        tgt, dft = _two_token_toy(gamma)
        T = 1.0
        acc = [so.acceptance_probability(so.row_probs(tgt[j], T), so.row_probs(dft[j], T), 0)
               for j in range(gamma)]
        surv, E = 1.0, 0.0
        for j in range(gamma):
            E += surv * (1 - acc[j]) * (j + 1)
            surv *= acc[j]
        E += surv * (gamma + 1)
        assert abs(E - oracle.expected_tokens_per_round(0.8, gamma)) < 1e-12


def tokens_per_round_mc(mod=so, rounds=20000, gamma=4, seed=7):
    tgt, dft = _two_token_toy(gamma)
    rng = np.random.default_rng(seed)
    counts = np.empty(rounds)
    for i in range(rounds):
        res = mod.verify_sample_seq(tgt, dft, [0] * gamma, 1.0, rng.random(gamma), rng.random())
        counts[i] = res.n + 1
        assert res.tokens[res.n] in (0, 1)
        if res.n < gamma:
            assert res.tokens[res.n] == 1  # residual of (0.8,0.2) vs (1,0) is token 1
    return counts


def test_tokens_per_round_monte_carlo_uniform_path():
    """The uniform-consuming path reproduces E = 3.3616 at alpha=0.8, gamma=4."""
    c = tokens_per_round_mc()
    E = oracle.expected_tokens_per_round(0.8, 4)
    se = c.std(ddof=1) / math.sqrt(len(c))
    assert abs(c.mean() - E) < 4 * se


def first_token_chi2(mod=so, V=8, rounds=20000, seed=13):
    """Empirical law of the first emitted token vs p_0 (chi-square statistic)."""
    rng = np.random.default_rng(seed)
    lt = rng.normal(0, 1.5, (2, V))
    ld = lt[:1] + rng.normal(0, 1.0, (1, V))
    p0 = so.row_probs(lt[0], 1.0)
    q0 = so.row_probs(ld[0], 1.0)
    counts = np.zeros(V)
    for _ in range(rounds):
        d = int(rng.choice(V, p=q0))
        res = mod.verify_sample_seq(lt, ld, [d], 1.0, [rng.random()], rng.random())
        counts[res.tokens[0]] += 1
    expct = rounds * p0
    return float(np.sum((counts - expct) ** 2 / expct))


def test_first_token_law_monte_carlo():
    # chi-square with 7 dof: P(X > 29) ~ 1.4e-4
    assert first_token_chi2() < 29.0


# ---------------------------------------------------------------------------
# residual identities, inverse CDF, decisions
# ---------------------------------------------------------------------------
def test_residual_identities():
    """P(accept x) = min(p, q) and the residual restores p exactly
    ("自投机解码…" §3.2)."""
    rng = np.random.default_rng(3)
    for V in (2, 8, 1000):
        p = so.row_probs(rng.normal(0, 2, V), 1.0)
        q = so.row_probs(rng.normal(0, 2, V), 1.0)
        w = so.residual_weights(p, q)
        Z = w.sum()
        accept_mass = np.minimum(p, q)
        assert abs(accept_mass.sum() + Z - 1.0) < 1e-13
        assert np.max(np.abs(accept_mass + Z * (w / Z) - p)) < 1e-15
        # rejection probability = sum_x q(x) (1 - min(1, p/q)) = Z
        rej = math.fsum(q[x] * (1 - so.acceptance_probability(p, q, x)) for x in range(V))
        assert abs(rej - Z) < 1e-13


def _icdf_bruteforce(w, u):
    """Definition written as a loop: the smallest k whose running total exceeds u*Z."""
    total = math.fsum(w)
    run = 0.0
    for k, x in enumerate(w):
        run += x
        if run > u * total:
            return k
    return max(i for i, x in enumerate(w) if x > 0)


def test_inverse_cdf_hand_cases():
    w = np.array([0.0, 0.25, 0.0, 0.75])
    assert so.inverse_cdf(w, 0.0)[0] == 1
    assert so.inverse_cdf(w, 0.2499)[0] == 1
    assert so.inverse_cdf(w, 0.25)[0] == 3       # C(1) = 0.25 is not > 0.25
    assert so.inverse_cdf(w, 0.3)[0] == 3
    assert so.inverse_cdf(w, 0.999999)[0] == 3
    k, m = so.inverse_cdf(w, 0.3)
    assert abs(m - 0.05) < 1e-15


def test_inverse_cdf_matches_bruteforce():
    rng = np.random.default_rng(17)
    for _ in range(300):
        V = int(rng.integers(1, 40))
        w = rng.random(V) * (rng.random(V) < 0.7)
        if w.sum() == 0:
            w[rng.integers(V)] = 1.0
        u = float(rng.random())
        assert so.inverse_cdf(w, u)[0] == _icdf_bruteforce(w, u)


def test_accept_decision_is_strict_u_below_ratio():
    lt = np.log(np.array([[0.3, 0.7], [0.5, 0.5]]))
    ld = np.log(np.array([[0.6, 0.4]]))
    rho = 0.3 / 0.6
    below = so.verify_sample_seq(lt, ld, [0], 1.0, [np.nextafter(rho, 0)], 0.1)
    at = so.verify_sample_seq(lt, ld, [0], 1.0, [rho], 0.1)
    assert below.n == 1 and at.n == 0
    assert at.tokens[0] == 1          # residual max(0, p-q) = (0, 0.3)


def test_special_cases():
    rng = np.random.default_rng(23)
    V, gamma = 64, 5
    lt = rng.normal(0, 2, (gamma + 1, V))
    # draft logits equal to target: rho = 1 -> all accepted, bonus drawn from p_gamma
    d = [int(x) for x in rng.integers(0, V, gamma)]
    u = rng.random(gamma) * 0.999
    res = so.verify_sample_seq(lt, lt[:gamma], d, 0.8, u, 0.37)
    assert res.n == gamma and res.path == "bonus"
    assert res.tokens[gamma] == _icdf_bruteforce(so.row_probs(lt[gamma], 0.8), 0.37)
    # one-hot target (other entries masked) at a != d: rejected, residual is delta_a
    one_hot = np.full((gamma + 1, V), -np.inf)
    one_hot[:, 9] = 0.0
    res = so.verify_sample_seq(one_hot, lt[:gamma], [3] * gamma, 1.0, [0.0] * gamma, 0.5)
    assert res.n == 0 and res.tokens[0] == 9
    # greedy: draft = argmax chain -> n = gamma, bonus = argmax of row gamma
    dg = [int(np.argmax(lt[j])) for j in range(gamma)]
    res = so.verify_greedy_seq(lt, dg)
    assert res.n == gamma and res.tokens[gamma] == int(np.argmax(lt[gamma]))
    # temperature <= 0 in the sampling entry is a greedy sequence
    res2 = so.verify_sample_seq(lt, lt[:gamma], dg, 0.0, u, 0.5)
    assert res2.tokens == res.tokens and res2.path == "greedy"


# ---------------------------------------------------------------------------
# the lm_head product against a brute-force loop
# ---------------------------------------------------------------------------
def test_lmhead_logits_bruteforce():
    rng = np.random.default_rng(29)
    R, V, H = 3, 5, 7
    h = rng.normal(0, 1, (R, H)).astype(np.float32)
    W = rng.normal(0, 0.02, (V, H)).astype(np.float32)
    got = so.lmhead_logits(h, W)
    for r in range(R):
        for x in range(V):
            want = math.fsum(float(h[r, k]) * float(W[x, k]) for k in range(H))
            assert abs(got[r, x] - want) < 1e-15


def test_lmhead_verify_groups_rows_per_sequence():
    """With W the identity (V = H) the lm_head logits are the hidden rows
    themselves, so the fused verify must reduce to plain sampling verification
    with target[b, j] = hidden[b*(gamma+1) + j]: pins the row grouping."""
    rng = np.random.default_rng(31)
    B, gamma, V = 3, 2, 8
    hidden = rng.normal(0, 2, (B * (gamma + 1), V))
    W = np.eye(V)
    target = hidden.reshape(B, gamma + 1, V)
    draft = target[:, :gamma] + rng.normal(0, 0.5, (B, gamma, V))
    toks = rng.integers(0, V, (B, gamma)).astype(np.int32)
    temp = np.array([1.0, 0.7, 0.0])
    ua = rng.random((B, gamma))
    ur = rng.random(B)
    got = so.verify_lmhead_sample(hidden, W, draft, toks, temp, ua, ur, gamma)
    want = so.verify_sample(target, draft, toks, temp, ua, ur)
    for g_, w_ in zip(got, want):
        assert g_.tokens == w_.tokens and g_.n == w_.n and g_.path == w_.path
        assert np.allclose(g_.L_p, w_.L_p, rtol=0, atol=1e-12)
    # a second W (a permutation) permutes the vocabulary of the target rows only
    perm = rng.permutation(V)
    got2 = so.verify_lmhead_sample(hidden, W[perm], draft, toks, temp, ua, ur, gamma)
    want2 = so.verify_sample(target[:, :, perm], draft, toks, temp, ua, ur)
    assert [r.tokens for r in got2] == [r.tokens for r in want2]


# ---------------------------------------------------------------------------
# speed-up model (host-side closed forms printed on the pages)
# ---------------------------------------------------------------------------
def test_speedup_closed_forms_printed_values():
    g = _golden("closed_forms.json")
    cf = g["cost_factor"]
    assert abs((1 + cf["gamma"] * cf["c"]) - cf["printed_value"]) < 1e-12
    s = g["speedup_naive"]
    for pt in s["points"]:
        assert round(oracle.speedup_naive(pt["alpha"], s["gamma"], s["c"]), 2) == pt["printed_value"]
    gain = oracle.speedup_naive(0.9, 4, 0.02) - oracle.speedup_naive(0.8, 4, 0.02)
    assert round(gain, 1) == s["gain_0p8_to_0p9_printed"]
    sw = g["speedup_layer_skip_sweep"]
    lo = [oracle.speedup_layer_skip(sw["alpha_low"], k, sw["c"]) for k in range(1, 11)]
    assert all(a > b for a, b in zip(lo, lo[1:]))
    gstar = oracle.best_gamma(sw["alpha_high"], sw["c"])
    assert sw["best_gamma_range"][0] <= gstar <= sw["best_gamma_range"][1]


# ---------------------------------------------------------------------------
# planted mistakes: each plausible error must fail one of the pins above
# ---------------------------------------------------------------------------
def test_mutation_residual_sign_is_caught(monkeypatch):
    monkeypatch.setattr(so, "residual_weights", lambda p, q: np.maximum(0.0, q - p))
    assert lossless_enumeration_error() > 1e-3


def test_mutation_inverted_ratio_is_caught(monkeypatch):
    def bad(p, q, d):
        return 1.0 if p[d] == 0 else min(1.0, float(q[d] / p[d]))
    monkeypatch.setattr(so, "acceptance_probability", bad)
    assert lossless_enumeration_error() > 1e-3


def test_mutation_dropped_temperature_is_caught(monkeypatch):
    orig = so.row_probs
    monkeypatch.setattr(so, "row_probs", lambda x, T: orig(x, 1.0))
    assert lossless_enumeration_error(T=0.6) > 1e-3


def test_mutation_row_offset_is_caught():
    def shifted(target_rows, draft_tokens):
        t = np.asarray(target_rows, dtype=np.float64)
        rolled = np.concatenate([t[1:], t[-1:]])   # verify d_{j+1} against row j+1
        return so.verify_greedy_seq(rolled, draft_tokens)
    assert greedy_chain_mismatches(shifted) > 0


def test_mutation_no_bonus_is_caught():
    def no_bonus(target_rows, draft_tokens):
        r = so.verify_greedy_seq(target_rows, draft_tokens)
        if r.n == len(draft_tokens):
            r.tokens[-1] = -1
            r.n -= 1   # the all-accepted branch emits nothing extra
        return r
    assert worked_example_failures(no_bonus) > 0


def test_mutation_wrong_uniform_compare_is_caught(monkeypatch):
    orig = so.verify_sample_seq

    def flipped(tp, tq, d, T, ua, ur):
        # reflect u about rho = 0.8 (the toy's ratio): accepts iff u > rho
        return orig(tp, tq, d, T, [1.6 - u for u in ua], ur)
    monkeypatch.setattr(so, "verify_sample_seq", flipped)
    # accept iff u > rho instead of u < rho: the mean count moves far from 3.3616
    c = tokens_per_round_mc(mod=so, rounds=4000)
    assert abs(c.mean() - oracle.expected_tokens_per_round(0.8, 4)) > 0.2


def test_mutation_icdf_off_by_one_is_caught(monkeypatch):
    orig = so.inverse_cdf

    def shifted(w, u):
        k, m = orig(w, u)
        return min(k + 1, len(w) - 1), m
    monkeypatch.setattr(so, "inverse_cdf", shifted)
    assert first_token_chi2(mod=so, rounds=5000) > 29.0


def test_mutation_multi_candidate_rules_are_caught(monkeypatch):
    """Keeping the shortest candidate, or the last of equal ones, fails a pin."""
    def shortest(target, draft_tokens):
        out = []
        for b in range(len(draft_tokens)):
            res = [so.verify_greedy_seq(target[b][c], draft_tokens[b][c]) for c in range(len(draft_tokens[b]))]
            best = min(range(len(res)), key=lambda c: res[c].n)
            out.append((res[best], best))
        return out
    assert multi_candidate_failures(shortest) > 0

    def last_of_equal(target, draft_tokens):
        out = []
        for b in range(len(draft_tokens)):
            res = [so.verify_greedy_seq(target[b][c], draft_tokens[b][c]) for c in range(len(draft_tokens[b]))]
            best = max(range(len(res)), key=lambda c: (res[c].n, c))
            out.append((res[best], best))
        return out
    monkeypatch.setattr(so, "verify_greedy_multi", last_of_equal)
    with pytest.raises(AssertionError):
        test_multi_candidate_ties_and_single_candidate()


# ---------------------------------------------------------------------------
# host round bookkeeping ("自投机解码…" §3.3; "Gemma 4 MTP 深度解析" §5.1)
# ---------------------------------------------------------------------------
def test_round_update_against_an_explicit_kv_cache():
    """Simulate the cache as a list of token ids: the verify pass appends the
    newest token and the gamma drafts, the rejected tail is dropped.  After
    every round the cache must hold exactly the sequence minus its newest
    token, and the oracle's kept length must equal the simulated one."""
    rng = np.random.default_rng(13)
    for trial in range(50):
        seq = list(rng.integers(0, 100, int(rng.integers(1, 20))))
        cache = seq[:-1]
        st = oracle.RoundState(gamma=int(rng.integers(1, 9)), seq_len=len(seq), kv_len=len(cache))
        for _ in range(30):
            g = st.gamma
            drafts = list(rng.integers(0, 100, g))
            n = int(rng.integers(0, g + 1))
            cache = cache + [seq[-1]] + drafts          # the verify pass
            emitted = drafts[:n] + [int(rng.integers(0, 100))]
            cache = cache[:len(seq) + n]                # drop entries of rejected drafts
            seq = seq + emitted
            keep = oracle.round_update(st, n, 1, 10)
            assert keep == len(cache) == st.kv_len and st.seq_len == len(seq)
            assert cache == seq[:-1]


def test_round_update_gamma_schedule_and_errors():
    st = oracle.RoundState(gamma=4, seq_len=7, kv_len=6)
    oracle.round_update(st, 4, 1, 10)   # every draft accepted: +2
    assert st.gamma == 6
    oracle.round_update(st, 2, 1, 10)   # a rejection: -1
    assert st.gamma == 5
    for _ in range(5):
        oracle.round_update(st, st.gamma, 1, 10)
    assert st.gamma == 10               # capped
    for _ in range(20):
        oracle.round_update(st, 0, 1, 10)
    assert st.gamma == 1                # floored
    with pytest.raises(ValueError):
        oracle.round_update(st, 2, 1, 10)          # more accepted than drafted
    bad = oracle.RoundState(gamma=4, seq_len=7, kv_len=7)
    with pytest.raises(ValueError):
        oracle.round_update(bad, 1, 1, 10)         # cache and sequence disagree


# ---------------------------------------------------------------------------
# top-k / top-p truncation ("Gemma 4 MTP 深度解析" §5.1: top_k=64, top_p=0.95;
# "第 8 章…" 为什么输出不会变: target and draft transformed the same way)
# ---------------------------------------------------------------------------
def _hf_truncate(l, T, k, top_p):
    """An independent formulation for distinct logits: keep the k largest
    scores; sort ascending, drop tokens whose cumulative softmax is <= 1 -
    top_p (the largest always stays); softmax of what is left."""
    z = np.asarray(l, np.float64) / T
    kth = np.sort(z)[::-1][min(k, len(z)) - 1]
    z = np.where(z < kth, -np.inf, z)
    order = np.argsort(z)
    pz = scipy.special.softmax(z[order])
    drop = np.cumsum(pz) <= 1 - top_p
    drop[-1] = False
    zz = z.copy()
    zz[order[drop]] = -np.inf
    return scipy.special.softmax(zz)


def test_truncate_topk_counts_and_ties():
    rng = np.random.default_rng(43)
    l = rng.normal(0, 2, 200)
    for k in (1, 5, 64, 199, 200, 500):
        p, _ = so.truncate_probs(l, 1.0, k, 1.0)
        assert (p > 0).sum() == min(k, 200)
        top = np.argsort(-l)[:min(k, 200)]
        assert set(np.flatnonzero(p)) == set(top)
    p, _ = so.truncate_probs(np.array([3.0, 1.0, 1.0, 1.0, 0.0]), 1.0, 2, 1.0)
    assert list(p > 0) == [True, True, True, True, False]     # the tie at the 2nd value stays
    assert abs(p.sum() - 1.0) < 1e-15


def test_truncate_topp_dyadic_boundaries():
    l = np.log([0.5, 0.25, 0.125, 0.125])                     # exact masses
    keep = lambda tp: list(so.truncate_probs(l, 1.0, 10, tp)[0] > 0)
    assert keep(0.5) == [True, False, False, False]           # mass above 0.25 is 0.5: not < 0.5
    assert keep(0.51) == [True, True, False, False]
    assert keep(0.75) == [True, True, False, False]           # mass above the 0.125s is 0.75
    assert keep(0.76) == [True, True, True, True]             # the tie group enters together
    assert keep(1e-9) == [True, False, False, False]          # the most likely token always stays
    p, m = so.truncate_probs(l, 1.0, 10, 0.75)
    assert abs(p[0] - 2 / 3) < 1e-15 and abs(m) < 1e-15       # the cut sits exactly on 0.75


def test_truncate_matches_an_independent_formulation():
    rng = np.random.default_rng(47)
    for _ in range(300):
        V = int(rng.integers(2, 300))
        l = rng.normal(0, float(rng.uniform(0.3, 4)), V)
        T = float(rng.uniform(0.3, 1.5))
        k = int(rng.integers(1, V + 5))
        tp = float(rng.uniform(0.05, 1.0))
        p, m = so.truncate_probs(l, T, k, tp)
        if m < 1e-9:
            continue
        assert np.allclose(p, _hf_truncate(l, T, k, tp), rtol=0, atol=1e-12)


def test_truncation_depends_on_temperature():
    l = np.log([0.5, 0.25, 0.125, 0.125])
    hot, _ = so.truncate_probs(l, 2.0, 10, 0.75)               # flatter: more tokens needed
    cold, _ = so.truncate_probs(l, 1.0, 10, 0.75)
    assert (hot > 0).sum() > (cold > 0).sum()


def _truncated_module(k, tp):
    import types
    m = types.SimpleNamespace()
    m.row_probs = lambda logits, T: so.truncate_probs(logits, T, k, tp)[0]
    m.acceptance_probability = so.acceptance_probability
    m.residual_weights = so.residual_weights
    return m


@pytest.mark.parametrize("k,tp", [(3, 1.0), (8, 0.7), (4, 0.9)])
def test_truncated_verification_is_lossless_V8(k, tp):
    """With p and q truncated the same way, the emitted tokens follow the
    truncated target distribution exactly (enumeration, V=8, gamma=2)."""
    mod = _truncated_module(k, tp)
    lm = ToyLM(V=8, salt=5, sd=1.2, draft_noise=1.0)
    T = 0.9

    @lru_cache(maxsize=None)
    def first_k(prefix, kk):
        out = {}
        for seq, w in _round_distribution(lm, list(prefix), 2, T, mod).items():
            if len(seq) >= kk:
                out[seq[:kk]] = out.get(seq[:kk], 0.0) + w
            else:
                for rest, w2 in first_k(prefix + seq, kk - len(seq)).items():
                    out[seq + rest] = out.get(seq + rest, 0.0) + w * w2
        return out

    spec = first_k((1,), 3)
    err = 0.0
    for t1 in range(8):
        p1 = _hf_truncate(lm.target_logits([1]), T, k, tp)[t1]
        for t2 in range(8):
            p2 = _hf_truncate(lm.target_logits([1, t1]), T, k, tp)[t2]
            for t3 in range(8):
                p3 = _hf_truncate(lm.target_logits([1, t1, t2]), T, k, tp)[t3]
                err = max(err, abs(spec.get((t1, t2, t3), 0.0) - p1 * p2 * p3))
    assert err < 1e-12


def test_mutation_topp_non_strict_is_caught(monkeypatch):
    orig = so.truncate_probs

    def non_strict(logits, temperature, top_k, top_p):
        return orig(logits, temperature, top_k, np.nextafter(top_p, 2.0))  # keeps "== top_p" too
    monkeypatch.setattr(so, "truncate_probs", non_strict)
    with pytest.raises(AssertionError):
        test_truncate_topp_dyadic_boundaries()


# ---------------------------------------------------------------------------
# centroid-masked sparse draft head and verification against its sparse q
# ("Gemma 4 MTP 深度解析" §3.4 Centroids Masking; "Gemma 4 - Drafter 解析", 高效 Embedder)
# ---------------------------------------------------------------------------
def _brute_head(h, C, W, off, o2t, top_k):
    """Explicit loops: fsum dot products, a Python sort by (-score, index)."""
    out = []
    for r in range(len(h)):
        z = [math.fsum(float(h[r][k]) * float(C[c][k]) for k in range(len(h[r]))) for c in range(len(C))]
        sel = sorted(range(len(C)), key=lambda c: (-z[c], c))[:top_k]
        cand = []
        for c in sel:
            for i in range(int(off[c]), int(off[c + 1])):
                cand.append((int(o2t[i]), math.fsum(float(h[r][k]) * float(W[i][k]) for k in range(len(h[r])))))
        cand.sort()
        out.append(cand)
    return out


def _tiny_centroid(seed=5, V=64, H=8, Nc=8):
    rng = np.random.default_rng(seed)
    cl = rng.integers(0, Nc, V)
    o2t = np.lexsort((np.arange(V), cl))
    off = np.concatenate([[0], np.cumsum(np.bincount(cl, minlength=Nc))])
    W = rng.normal(0, 1, (V, H))
    C = rng.normal(0, 1, (Nc, H))
    h = rng.normal(0, 1, (3, H))
    return h, C, W, off, o2t


def test_centroid_head_matches_brute_force():
    h, C, W, off, o2t = _tiny_centroid()
    for top_k in (1, 3, 8):
        got = oracle.centroid_head(h, C, W, off, o2t, top_k)
        want = _brute_head(h, C, W, off, o2t, top_k)
        for (tok, lg), cand in zip(got, want):
            assert list(tok) == [t for t, _ in cand]
            assert np.allclose(lg, [x for _, x in cand], rtol=0, atol=1e-12)


def test_centroid_head_all_clusters_is_the_dense_head():
    h, C, W, off, o2t = _tiny_centroid(seed=6, V=96, H=6, Nc=7)
    dense = oracle.lmhead_logits(h, W[np.argsort(o2t)])  # token order
    for r, (tok, lg) in enumerate(oracle.centroid_head(h, C, W, off, o2t, 7)):
        assert list(tok) == list(range(96))
        assert np.allclose(lg, dense[r], rtol=0, atol=1e-12)


def test_centroid_top_clusters_ties_keep_the_lowest_index():
    assert list(oracle.top_clusters([1.0, 3.0, 3.0, 2.0, 3.0], 2)) == [1, 2]
    assert list(oracle.top_clusters([0.5, 0.5, 0.5], 3)) == [0, 1, 2]
    h, C, W, off, o2t = _tiny_centroid(seed=8)
    C[5] = C[2]  # clusters 2 and 5 score the same for every row
    z = oracle.cluster_scores(h, C)
    for r in range(len(h)):
        sel = list(oracle.top_clusters(z[r], 8))
        assert sel.index(2) < sel.index(5)


def test_sparse_row_to_dense_gives_the_candidate_softmax():
    tok = np.array([1, 4, 6])
    lg = np.array([0.5, -1.0, 2.0])
    row = oracle.sparse_row_to_dense(tok, lg, 8)
    q = oracle.row_probs(row, 0.7)
    want = scipy.special.softmax(lg / 0.7)
    assert np.allclose(q[tok], want, rtol=0, atol=1e-15)
    assert q[[0, 2, 3, 5, 7]].sum() == 0.0


class _MaskedDraftLM(ToyLM):
    """q restricted to the 3 tokens with the largest draft logits (q = 0 elsewhere)."""

    def draft_logits(self, prefix):
        l = super().draft_logits(prefix)
        keep = np.argsort(-l, kind="stable")[:3]
        tok = np.sort(keep)
        return oracle.sparse_row_to_dense(tok, l[tok], self.V)


def test_sparse_draft_verification_is_lossless_V8():
    lm = _MaskedDraftLM(V=8, salt=11, sd=1.2, draft_noise=1.0)
    T = 0.9

    @lru_cache(maxsize=None)
    def first_k(prefix, kk):
        out = {}
        for seq, w in _round_distribution(lm, list(prefix), 2, T, so).items():
            if len(seq) >= kk:
                out[seq[:kk]] = out.get(seq[:kk], 0.0) + w
            else:
                for rest, w2 in first_k(prefix + seq, kk - len(seq)).items():
                    out[seq + rest] = out.get(seq + rest, 0.0) + w * w2
        return out

    spec = first_k((2,), 3)
    err = 0.0
    for t1 in range(8):
        p1 = scipy.special.softmax(lm.target_logits([2]) / T)[t1]
        for t2 in range(8):
            p2 = scipy.special.softmax(lm.target_logits([2, t1]) / T)[t2]
            for t3 in range(8):
                p3 = scipy.special.softmax(lm.target_logits([2, t1, t2]) / T)[t3]
                err = max(err, abs(spec.get((t1, t2, t3), 0.0) - p1 * p2 * p3))
    assert err < 1e-12


def test_verify_sample_sparse_full_candidates_is_verify_sample():
    import workloads as wl
    m = wl.make_centroid_model(V=2048, H=32, n_clusters=16, seed=3, mu_sd=0.3, eps_sd=0.05)
    rd = wl.make_centroid_round(m, B=6, gamma=3, r=1, draft_sd=0.1, temperature=0.8)
    cand = oracle.centroid_head(rd["hidden_draft"], m.centroids, m.W_ord, m.cluster_off, m.ord2tok, 16)
    d = wl.sample_sparse_drafts(cand, rd["temperature"], 3, r=1)
    dense = oracle.lmhead_logits(rd["hidden_draft"], m.W_ord[m.tok2ord]).reshape(6, 3, -1)
    got = oracle.verify_sample_sparse(rd["target"], [[cand[b * 3 + j] for j in range(3)] for b in range(6)], d,
                                      rd["temperature"], rd["u_accept"], rd["u_resample"])
    want = oracle.verify_sample(rd["target"], dense, d, rd["temperature"], rd["u_accept"], rd["u_resample"])
    for a, b in zip(got, want):
        assert a.n == b.n and a.tokens == b.tokens


def test_mutation_centroid_rules_are_caught(monkeypatch):
    """Highest index on ties, or a cluster range one row short, fails a pin."""
    import oracle.centroid as oc
    orig_top = oc.top_clusters
    highest = lambda s, k: np.lexsort((-np.arange(len(s)), -np.asarray(s)))[:k]
    monkeypatch.setattr(oc, "top_clusters", highest)
    monkeypatch.setattr(oracle, "top_clusters", highest)
    with pytest.raises(AssertionError):
        test_centroid_top_clusters_ties_keep_the_lowest_index()
    monkeypatch.setattr(oc, "top_clusters", orig_top)
    monkeypatch.setattr(oracle, "top_clusters", orig_top)
    orig_head = oc.centroid_head

    def short_range(hidden, centroids, W_ord, cluster_off, ord2tok, top_k):
        off = np.asarray(cluster_off).copy()
        off[1:] = np.maximum(off[1:] - 1, off[:-1])
        return orig_head(hidden, centroids, W_ord, off, ord2tok, top_k)
    monkeypatch.setattr(oracle, "centroid_head", short_range)
    with pytest.raises(AssertionError):
        test_centroid_head_matches_brute_force()


def test_mutation_sparse_fill_is_caught(monkeypatch):
    """Non-candidates filled with logit 0 instead of -inf gives q > 0 off the
    candidates: the softmax pin fails."""
    orig = oracle.sparse_row_to_dense
    monkeypatch.setattr(oracle, "sparse_row_to_dense",
                        lambda t, l, V: np.where(np.isin(np.arange(V), t), orig(t, l, V), 0.0))
    with pytest.raises(AssertionError):
        test_sparse_row_to_dense_gives_the_candidate_softmax()


def test_verify_sample_sparse_empty_rows_accept_every_draft():
    """No candidates: q = 0 everywhere, every draft is accepted (q(d) = 0) and
    the bonus is the inverse CDF of p_gamma with the resample uniform."""
    rng = np.random.default_rng(13)
    V, gamma = 64, 3
    target = rng.normal(0, 1.5, (1, gamma + 1, V))
    empty = (np.zeros(0, np.int64), np.zeros(0))
    res = oracle.verify_sample_sparse(target, [[empty] * gamma], np.array([[5, 9, 60]]), np.array([0.9]),
                                      np.array([[0.999, 0.5, 0.0]]), np.array([0.37]))
    r = res[0]
    assert r.n == gamma and r.tokens[:gamma] == [5, 9, 60]
    p = scipy.special.softmax(target[0, gamma] / 0.9)
    assert r.tokens[gamma] == int(np.searchsorted(np.cumsum(p), 0.37, side="right"))


# ---------------------------------------------------------------------------
# the excusal margins.  A GPU result that differs from the oracle is excused
# only where the oracle's margin is below the agreed window, so each margin is
# pinned by what it promises, not by its formula: moving any one uniform (or
# top_p) that took part in a decision by less than the margin leaves the
# output unchanged, and moving one of them a little further than the margin,
# towards the boundary it is nearest to, changes it.
# ("Gemma 4 Multi-Token Prediction (MTP) 深度解析" §2.2: accept with
# probability min(1, p/q); the stated 1e-6 window on uniforms near a boundary)
# ---------------------------------------------------------------------------
def _margin_cases(n, seed):
    """Small random sequences: V in [3, 40], gamma in [1, 5], T in [0.4, 1.6],
    draft logits = target + noise, drafts drawn from q."""
    rng = np.random.default_rng(seed)
    for _ in range(n):
        V = int(rng.integers(3, 41))
        g = int(rng.integers(1, 6))
        T = float(rng.uniform(0.4, 1.6))
        lt = rng.normal(0, 1.5, (g + 1, V))
        ld = lt[:g] + rng.normal(0, float(rng.uniform(0.2, 1.5)), (g, V))
        d = [int(rng.choice(V, p=scipy.special.softmax(ld[j] / T))) for j in range(g)]
        yield lt, ld, d, T, rng.random(g), float(rng.random())


def _same(a, b):
    return a.n == b.n and a.tokens == b.tokens


def margin_flip_violations(mod=so, n=400, seed=101):
    """Cases where a SeqResult's margin breaks its promise (see above)."""
    bad = 0
    for lt, ld, d, T, ua, ur in _margin_cases(n, seed):
        base = mod.verify_sample_seq(lt, ld, d, T, ua, ur)
        m = base.margin
        if not (0.0 < m < math.inf):
            continue
        # the uniforms that took part: u_accept[0..n] and u_resample
        slots = [("a", j) for j in range(min(base.n + 1, len(d)))] + [("r", 0)]

        def moved(slot, delta):
            """The output with one uniform moved, or None when that takes the
            resample uniform out of [0, 1), where the draw is not defined."""
            a, r = list(ua), ur
            if slot[0] == "a":
                a[slot[1]] += delta     # u < rho is defined for any real u
            else:
                r += delta
                if not 0.0 <= r < 1.0:
                    return None
            return mod.verify_sample_seq(lt, ld, d, T, a, r)

        near = [moved(s, sgn * m * (1 - 1e-7)) for s in slots for sgn in (1, -1)]
        far = [moved(s, sgn * (m * (1 + 1e-7) + 1e-15)) for s in slots for sgn in (1, -1)]
        far = [r for r in far if r is not None]
        inside = all(r is None or _same(base, r) for r in near)
        beyond = not far or any(not _same(base, r) for r in far)
        bad += (not inside) + (not beyond)
    return bad


def test_sample_margin_keeps_its_promise():
    assert margin_flip_violations() == 0


def test_acceptance_margin_hand_cases():
    """rho = p(d)/q(d) = 0.5 exactly (dyadic rows): u sits 2^-20 from it."""
    lt = np.log(np.array([[0.25, 0.75], [0.5, 0.5]]))
    ld = np.log(np.array([[0.5, 0.5]]))
    for u, accepted in ((0.5 - 2.0 ** -20, True), (0.5 + 2.0 ** -20, False)):
        res = so.verify_sample_seq(lt, ld, [0], 1.0, [u], 0.3)   # draw edges 0.2 away or more
        assert (res.n == 1) == accepted
        assert abs(res.margin - 2.0 ** -20) < 1e-15      # the accept boundary is the nearer one
    # a single token of residual weight: the draw has no boundary at all
    res = so.verify_sample_seq(lt, ld, [0], 1.0, [0.9], 0.3)
    assert res.n == 0 and res.tokens[0] == 1 and abs(res.margin - 0.4) < 1e-15
    # far from rho the interior CDF edge of the draw is the nearer boundary:
    # p = (1/8, 3/8, 1/2), q = (1/2, 1/4, 1/4), d = 0: rho = 1/4; after the
    # rejection w = (0, 1/8, 1/4), edge 1/3 between tokens 1 and 2
    lt3 = np.log(np.array([[0.125, 0.375, 0.5], [1 / 3, 1 / 3, 1 / 3]]))
    ld3 = np.log(np.array([[0.5, 0.25, 0.25]]))
    res = so.verify_sample_seq(lt3, ld3, [0], 1.0, [0.9], 0.3)
    assert res.n == 0 and res.tokens[0] == 1 and abs(res.margin - (1 / 3 - 0.3)) < 1e-15
    res = so.verify_sample_seq(lt3, ld3, [0], 1.0, [0.9], 0.34)
    assert res.tokens[0] == 2 and abs(res.margin - (0.34 - 1 / 3)) < 1e-15
    # rho >= 1 everywhere (q == p): the accept margins are rho - u = 1 - u
    res = so.verify_sample_seq(lt, lt[:1], [1], 1.0, [0.9999], 0.3)
    assert res.n == 1 and abs(res.margin - 1e-4) < 1e-12


def test_greedy_margin_is_infinite():
    lt = np.log(np.array([[0.25, 0.75], [0.5, 0.5]]))
    assert so.verify_greedy_seq(lt, [1]).margin == math.inf


def _kept(p):
    return tuple(np.flatnonzero(p > 0))


def topp_margin_violations(trunc=None, n=400, seed=103):
    """Rows where truncate_probs's margin breaks its promise: moving top_p by
    less than it keeps the kept set, moving it a little further (up or down)
    changes it."""
    trunc = trunc or so.truncate_probs
    rng = np.random.default_rng(seed)
    bad = 0
    for _ in range(n):
        V = int(rng.integers(2, 60))
        l = rng.normal(0, float(rng.uniform(0.3, 3.0)), V)
        T = float(rng.uniform(0.4, 1.6))
        k = int(rng.integers(1, V + 3))
        tp = float(rng.uniform(0.05, 0.99))
        p, m = trunc(l, T, k, tp)
        if not (0.0 < m < 1.0):
            continue
        base = _kept(p)
        # top_p moves only inside its domain (0, 1]
        near = [tp + s * m * (1 - 1e-7) for s in (1, -1)]
        far = [tp + s * (m * (1 + 1e-7) + 1e-15) for s in (1, -1)]
        inside = all(_kept(trunc(l, T, k, x)[0]) == base for x in near if 0.0 < x <= 1.0)
        far = [x for x in far if 0.0 < x <= 1.0]
        beyond = not far or any(_kept(trunc(l, T, k, x)[0]) != base for x in far)
        bad += (not inside) + (not beyond)
    return bad


def test_topp_margin_keeps_its_promise():
    assert topp_margin_violations() == 0


def test_topp_margin_hand_case():
    # masses (1/2, 1/4, 1/8, 1/8): the cuts sit at mass-above 0, 1/2, 3/4
    l = np.log([0.5, 0.25, 0.125, 0.125])
    for tp, m in ((0.6, 0.1), (0.74, 0.01), (0.3, 0.2), (0.95, 0.2), (0.1, 0.4)):
        assert abs(so.truncate_probs(l, 1.0, 10, tp)[1] - m) < 1e-15


def test_topkp_sequence_margin_covers_every_row():
    """The sequence-level trunc_margin: moving top_p by less than it leaves the
    whole verification unchanged."""
    rng = np.random.default_rng(107)
    for _ in range(60):
        V, g = int(rng.integers(4, 30)), int(rng.integers(1, 4))
        T = float(rng.uniform(0.5, 1.5))
        lt = rng.normal(0, 1.5, (g + 1, V))
        ld = lt[:g] + rng.normal(0, 0.7, (g, V))
        k, tp = int(rng.integers(2, V + 1)), float(rng.uniform(0.3, 0.95))
        d = [int(x) for x in rng.integers(0, V, g)]
        ua, ur = rng.random(g), float(rng.random())
        base = so.verify_sample_topkp_seq(lt, ld, d, T, k, tp, ua, ur)
        m = base.trunc_margin
        if not (0.0 < m < 1.0):
            continue
        for s in (1, -1):
            r = so.verify_sample_topkp_seq(lt, ld, d, T, k, tp + s * m * (1 - 1e-7), ua, ur)
            assert _same(base, r) and r.p_tok == base.p_tok and r.q_tok == base.q_tok
        # a little beyond it, some row's kept set changes
        rows = [lt[j] for j in range(g + 1)] + [ld[j] for j in range(g)]
        assert any(_kept(so.truncate_probs(x, T, k, tp + s * (m * (1 + 1e-7) + 1e-15))[0]) !=
                   _kept(so.truncate_probs(x, T, k, tp)[0]) for x in rows for s in (1, -1))


def test_mutation_relative_acceptance_margin_is_caught(monkeypatch):
    """|u - rho| / rho instead of |u - rho|."""
    orig = so._decide_and_draw

    def relative(P, Q, d, ua, ur, L_p, L_q):
        r = orig(P, Q, d, ua, ur, L_p, L_q)
        m = math.inf
        for j in range(min(r.n + 1, len(d))):
            rho = math.inf if r.q_tok[j] == 0 else r.p_tok[j] / r.q_tok[j]
            if rho != math.inf:
                m = min(m, abs(float(ua[j]) - rho) / rho)
        w = so.residual_weights(P[r.n], Q[r.n]) if r.n < len(d) else P[len(d)]
        r.margin = min(m, so.inverse_cdf(w, float(ur))[1])
        return r
    monkeypatch.setattr(so, "_decide_and_draw", relative)
    assert margin_flip_violations(n=200) > 0


def test_mutation_margin_of_the_wrong_decision_is_caught(monkeypatch):
    """Only the deciding position's distance (j = n), not the accepted ones before it."""
    orig = so._decide_and_draw

    def last_only(P, Q, d, ua, ur, L_p, L_q):
        r = orig(P, Q, d, ua, ur, L_p, L_q)
        j = min(r.n, len(d) - 1)
        rho = math.inf if r.q_tok[j] == 0 else r.p_tok[j] / r.q_tok[j]
        m = abs(float(ua[j]) - rho) if rho != math.inf else math.inf
        w = so.residual_weights(P[r.n], Q[r.n]) if r.n < len(d) else P[len(d)]
        r.margin = min(m, so.inverse_cdf(w, float(ur))[1])
        return r
    monkeypatch.setattr(so, "_decide_and_draw", last_only)
    assert margin_flip_violations(n=400) > 0


def test_mutation_one_sided_cdf_margin_is_caught(monkeypatch):
    """The distance to the upper CDF edge only."""
    def upper_only(w, u):
        c = np.cumsum(w)
        z = c[-1]
        k = int(np.searchsorted(c, u * z, side="right"))
        if k >= len(w):
            return int(np.flatnonzero(w > 0)[-1]), 0.0
        return k, float(c[k] / z - u)
    monkeypatch.setattr(so, "inverse_cdf", upper_only)
    assert margin_flip_violations(n=200) > 0


def test_mutation_topp_margin_below_the_cut_is_caught():
    """The mass up to and including a token, instead of strictly above it."""
    def below(logits, temperature, top_k, top_p):
        p, _ = so.truncate_probs(logits, temperature, top_k, top_p)
        l = np.asarray(logits, np.float64)
        order = np.argsort(-l, kind="stable")
        greater = np.searchsorted(-l[order], -l[order], side="left")
        idx_k = order[greater < top_k]
        zk = l[idx_k] / temperature
        pk = scipy.special.softmax(zk)
        upto = np.cumsum(pk)
        return p, float(np.min(np.abs(upto - top_p)))
    assert topp_margin_violations(trunc=below, n=200) > 0
