"""fp64 CPU oracle for the speculative-decoding verify-and-accept step.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain reference that the
CUDA path is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product library never imports, links or calls it, and it shares no code,
tables or helpers with the CUDA sources.

Everything is computed in float64 with numpy.  bf16 and fp32 inputs widen to
float64 exactly.  Each function cites the page and section it follows.  The
five source pages are:

* [MTP-blog]   "Accelerating Gemma 4: faster inference with multi-token
               prediction drafters" (zskr.cn), §3.2 验证与接受机制, §4.1.
* [Drafter]    "Gemma 4 - Drafter 解析" (easyvibecoding curated post).
* [MTP-deep]   "Gemma 4 Multi-Token Prediction (MTP) 深度解析", §2.2 推测解码的数学保证,
               §3.4 Centroids Masking.
* [Book-ch8]   "第 8 章 投机解码：一次前向，验证好几个字", sections 先看一个具体的例子,
               为什么输出不会变, 多出来的那一个 token 从哪来, 收益怎么算.
* [Self-spec]  "自投机解码：层跳过与拒绝采样实现大模型推理加速", §3.1 贪心解码,
               §3.2 采样解码, §3.3 随机数与 batch 内对齐, §4.1, §4.2.

Readings where the pages are silent:

* accept iff ``u < rho`` with ``u`` in [0, 1); ``q(d) == 0`` accepts.
* inverse CDF in ascending vocabulary order, strict ``>``: token
  ``k = min{k : C(k) > u * Z}``; if rounding leaves no such k, the last token
  with nonzero weight.
* the bonus token under sampling is drawn from ``p_gamma`` with the same
  per-sequence resample uniform (only one of residual / bonus happens).
* a residual with ``Z == 0`` (unreachable in exact arithmetic) samples from
  ``p_n`` instead.
* greedy rows (temperature <= 0) compare the draft with the argmax of the raw
  logits, lowest index on ties; the greedy replacement / bonus is that argmax.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, exhaustive enumeration, brute force, library routines).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "bf16_bits_to_f64",
    "row_log_normaliser",
    "row_probs",
    "row_argmax",
    "acceptance_probability",
    "residual_weights",
    "inverse_cdf",
    "SeqResult",
    "verify_greedy_seq",
    "verify_sample_seq",
    "verify_greedy",
    "verify_sample",
    "lmhead_logits",
    "verify_lmhead_sample",
    "verify_greedy_multi",
    "truncate_probs",
    "verify_sample_topkp_seq",
    "verify_sample_topkp",
]


# ---------------------------------------------------------------------------
# input widening
# ---------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 values stored as raw uint16 bit patterns to float64.

    A bf16 number is the upper half of an IEEE binary32 word, so shifting the
    16 bits into the top of a 32-bit word gives the same value as a float32,
    which float64 then holds exactly.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _as_f64(x) -> np.ndarray:
    """Logits in float64: uint16 arrays are bf16 bit patterns, floats widen."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return x.astype(np.float64)


# ---------------------------------------------------------------------------
# temperature softmax ([Book-ch8] 为什么输出不会变: temperature is applied the
# same way to draft and target; [Self-spec] §3.1: temperature 0 is greedy)
# ---------------------------------------------------------------------------
def row_log_normaliser(logits: np.ndarray, temperature: float) -> float:
    """L = ln sum_x exp(l_x / T), evaluated as M + ln sum exp(l/T - M)."""
    z = logits / temperature
    m = np.max(z)
    if m == -np.inf:
        return -np.inf
    return float(m + np.log(np.sum(np.exp(z - m))))


def row_probs(logits: np.ndarray, temperature: float) -> np.ndarray:
    """p_x = exp(l_x / T - L): the temperature softmax of one row."""
    return np.exp(logits / temperature - row_log_normaliser(logits, temperature))


def row_argmax(logits: np.ndarray) -> int:
    """Index of the largest raw logit; the lowest such index on ties."""
    top = np.max(logits)
    return int(np.flatnonzero(logits == top)[0])


# ---------------------------------------------------------------------------
# rejection sampling pieces ([MTP-deep] §2.2; [Book-ch8] 为什么输出不会变;
# [Self-spec] §3.2)
# ---------------------------------------------------------------------------
def acceptance_probability(p: np.ndarray, q: np.ndarray, d: int) -> float:
    """min(1, p(d) / q(d)); a draft the drafter gave zero mass is accepted."""
    if q[d] == 0.0:
        return 1.0
    return min(1.0, float(p[d] / q[d]))


def residual_weights(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Unnormalised corrected distribution w = max(0, p - q)."""
    return np.maximum(0.0, p - q)


def inverse_cdf(w: np.ndarray, u: float) -> tuple[int, float]:
    """Sample index k = min{k : C(k) > u * Z}, C the running sum of w, Z = C(V-1).

    Returns (k, margin) where margin is the distance in u units from u to the
    nearer edge [C(k-1)/Z, C(k)/Z) of the chosen interval that another token
    lies beyond.  The outer edges 0 and Z are not decision boundaries: below
    the first token with weight nothing else can be drawn, and past the total
    the last token with weight is drawn, so an edge with no weight beyond it
    does not count.  When rounding leaves no index with C(k) > u*Z, the last
    index with w > 0 is taken and the margin is 0.
    """
    c = np.cumsum(w)
    z = c[-1]
    target = u * z
    k = int(np.searchsorted(c, target, side="right"))
    if k >= len(w):
        nz = np.flatnonzero(w > 0)
        return int(nz[-1]), 0.0
    lo = c[k - 1] if k > 0 else 0.0
    below = u - lo / z if lo > 0.0 else math.inf      # a token with weight lies below
    above = c[k] / z - u if c[k] < z else math.inf     # a token with weight lies above
    return k, float(min(below, above))


# ---------------------------------------------------------------------------
# one sequence
# ---------------------------------------------------------------------------
@dataclass
class SeqResult:
    """Outcome for one sequence.

    tokens: gamma+1 ints; the first n+1 are emitted, the rest are -1.
    n: number of accepted draft tokens (0..gamma).
    margin: the smallest distance, in uniform units, between a uniform that
        took part in a decision and the boundary it was compared with
        (inf for greedy).  A GPU result that differs from the oracle is
        excused only where this is below the agreed window.
    p_tok, q_tok: p_j(d_{j+1}) and q_j(d_{j+1}) for j < gamma (nan if greedy).
    L_p, L_q: ln-normalisers of target rows 0..gamma and draft rows 0..gamma-1.
    path: "greedy", "residual", "bonus" or "residual_z0".
    trunc_margin: with top-k / top-p truncation, the smallest distance (in
        probability mass) between a top-p cut and top_p (inf otherwise).
    """

    tokens: list
    n: int
    margin: float = math.inf
    p_tok: list = field(default_factory=list)
    q_tok: list = field(default_factory=list)
    L_p: list = field(default_factory=list)
    L_q: list = field(default_factory=list)
    path: str = "greedy"
    trunc_margin: float = math.inf


def verify_greedy_seq(target_rows, draft_tokens) -> SeqResult:
    """Greedy verification of one sequence.

    Row j of the target is its next-token distribution after prefix + d_1..d_j
    ([Book-ch8] 为什么一次前向能验证多个 token).  Draft d_{j+1} is accepted iff it
    is the target's argmax at row j ([MTP-blog] §3.2; [Self-spec] §3.1).  At
    the first mismatch n the target's own argmax replaces the draft
    ([Self-spec] §3.1); if every draft matches, row gamma gives one more token
    (the N+1 bonus, [Book-ch8] 多出来的那一个 token 从哪来).
    """
    t = _as_f64(target_rows)
    d = [int(x) for x in draft_tokens]
    gamma = len(d)
    assert t.shape[0] == gamma + 1
    n = gamma
    for j in range(gamma):
        if d[j] != row_argmax(t[j]):
            n = j
            break
    tokens = d[:n] + [row_argmax(t[n])] + [-1] * (gamma - n)
    return SeqResult(tokens=tokens, n=n, path="greedy")


def _decide_and_draw(P, Q, d, u_accept, u_resample, L_p, L_q) -> SeqResult:
    """The sampling decision on probability rows P[0..gamma], Q[0..gamma-1]:
    accept d_{j+1} iff u_accept[j] < P[j][d]/Q[j][d], stop at the first
    rejection n, then draw position n by inverse CDF from max(0, P[n] - Q[n])
    (from P[gamma] if every draft passed)."""
    gamma = len(d)
    p_tok, q_tok = [], []
    margin = math.inf
    n = gamma
    for j in range(gamma):
        p_tok.append(float(P[j][d[j]]))
        q_tok.append(float(Q[j][d[j]]))
    for j in range(gamma):
        # the decision compares u with the plain ratio p/q (inf when q = 0)
        rho = math.inf if q_tok[j] == 0.0 else p_tok[j] / q_tok[j]
        u = float(u_accept[j])
        if rho != math.inf:
            margin = min(margin, abs(u - rho))
        if not (u < rho):
            n = j
            break

    if n < gamma:
        w = residual_weights(P[n], Q[n])
        path = "residual"
        if not np.any(w > 0):
            w = P[n]
            path = "residual_z0"
    else:
        w = P[gamma]
        path = "bonus"
    tok, m2 = inverse_cdf(w, float(u_resample))
    margin = min(margin, m2)
    tokens = d[:n] + [tok] + [-1] * (gamma - n)
    return SeqResult(tokens=tokens, n=n, margin=margin, p_tok=p_tok,
                     q_tok=q_tok, L_p=L_p, L_q=L_q, path=path)


def verify_sample_seq(target_rows, draft_rows, draft_tokens, temperature,
                      u_accept, u_resample) -> SeqResult:
    """Rejection-sampling verification of one sequence.

    p_j = softmax(l_p[j] / T), q_j = softmax(l_q[j] / T).  Walking j = 0, 1, ...
    the draft d_{j+1} is accepted iff u_accept[j] < p_j(d)/q_j(d), i.e. with
    probability min(1, p/q) ([MTP-deep] §2.2; [Book-ch8] 为什么输出不会变;
    [Self-spec] §3.2).  The first rejection n stops the walk and the later
    drafts are discarded ([Self-spec] §2.1, §3.3).  Position n is then drawn
    from max(0, p_n - q_n) / Z by inverse CDF with u_resample; if all gamma
    drafts pass, it is drawn from p_gamma instead (the bonus token,
    [Book-ch8] 多出来的那一个 token 从哪来).  Each sequence brings its own uniforms
    ([Self-spec] §3.3).
    """
    T = float(temperature)
    if T <= 0.0:
        return verify_greedy_seq(target_rows, draft_tokens)
    tp = _as_f64(target_rows)
    tq = _as_f64(draft_rows)
    d = [int(x) for x in draft_tokens]
    gamma = len(d)
    assert tp.shape[0] == gamma + 1 and tq.shape[0] == gamma

    L_p = [row_log_normaliser(tp[j], T) for j in range(gamma + 1)]
    L_q = [row_log_normaliser(tq[j], T) for j in range(gamma)]
    P = [np.exp(tp[j] / T - L_p[j]) for j in range(gamma + 1)]
    Q = [np.exp(tq[j] / T - L_q[j]) for j in range(gamma)]
    return _decide_and_draw(P, Q, d, u_accept, u_resample, L_p, L_q)


# ---------------------------------------------------------------------------
# top-k / top-p truncation, applied identically to target and draft
# ([MTP-deep] §5.1: sampling with top_k=64, top_p=0.95 next to the drafter;
# [Book-ch8] 为什么输出不会变: whatever transforms the target distribution must
# transform the draft distribution the same way)
# ---------------------------------------------------------------------------
def truncate_probs(logits, temperature: float, top_k: int, top_p: float):
    """The truncated distribution of one row: returns (p, margin).

    K  = tokens with fewer than top_k strictly larger logits (ties at the k-th
         value stay in);
    pk = softmax(l / T) over K;
    K' = tokens x of K whose strictly more likely tokens in K hold less than
         top_p of pk (a tie group stays together; the most likely tokens are
         always kept);
    p  = softmax(l / T) over K', 0 elsewhere.
    margin = min over x in K below the most likely tie group of
    |mass strictly above x - top_p|: how far the top-p cut is from flipping
    (inf when top_p >= 1).  The most likely group (mass above it 0) is kept
    for every top_p > 0, so it sets no boundary.
    """
    l = _as_f64(logits)
    z = l / float(temperature)
    order = np.argsort(-l, kind="stable")          # descending; ties by index
    ls = l[order]
    # top-k with ties: keep x iff #{y : l_y > l_x} < k
    greater = np.searchsorted(-ls, -ls, side="left")   # count of strictly larger values
    in_k = greater < top_k
    idx_k = order[in_k]
    zk = z[idx_k]
    pk = np.exp(zk - (zk.max() + np.log(np.sum(np.exp(zk - zk.max())))))
    lk = l[idx_k]
    # mass strictly above each kept token (sorted descending, ties grouped)
    cum = np.concatenate([[0.0], np.cumsum(pk)])
    first = np.searchsorted(-lk, -lk, side="left")
    above = cum[first]
    keep = above < top_p
    cuts = above[above > 0.0]
    margin = math.inf if (top_p >= 1.0 or cuts.size == 0) else float(np.min(np.abs(cuts - top_p)))
    kept = idx_k[keep]
    p = np.zeros_like(l)
    zz = z[kept]
    m = zz.max()
    p[kept] = np.exp(zz - m - np.log(np.sum(np.exp(zz - m))))
    return p, margin


def verify_sample_topkp_seq(target_rows, draft_rows, draft_tokens, temperature,
                            top_k, top_p, u_accept, u_resample) -> SeqResult:
    """Rejection-sampling verification with both p_j and q_j truncated by
    ``truncate_probs`` (same T, top_k, top_p).  L_p, L_q are the ln
    normalisers of the truncated rows (ln of the sum of exp(l/T) over the
    kept tokens); ``trunc_margin`` is the smallest top-p cut margin of the
    rows used."""
    T = float(temperature)
    if T <= 0.0:
        return verify_greedy_seq(target_rows, draft_tokens)
    tp = _as_f64(target_rows)
    tq = _as_f64(draft_rows)
    d = [int(x) for x in draft_tokens]
    gamma = len(d)
    P, Q, L_p, L_q, tm = [], [], [], [], math.inf
    for j in range(gamma + 1):
        pj, mj = truncate_probs(tp[j], T, top_k, top_p)
        P.append(pj)
        kept = pj > 0
        L_p.append(row_log_normaliser(np.where(kept, tp[j], -np.inf), T))
        tm = min(tm, mj)
    for j in range(gamma):
        qj, mj = truncate_probs(tq[j], T, top_k, top_p)
        Q.append(qj)
        kept = qj > 0
        L_q.append(row_log_normaliser(np.where(kept, tq[j], -np.inf), T))
        tm = min(tm, mj)
    res = _decide_and_draw(P, Q, d, u_accept, u_resample, L_p, L_q)
    res.trunc_margin = tm
    return res


# ---------------------------------------------------------------------------
# batches: sequences are independent ([Self-spec] §3.3: per-sequence counts)
# ---------------------------------------------------------------------------
def verify_greedy(target, draft_tokens) -> list[SeqResult]:
    """target [B, gamma+1, V]; draft_tokens [B, gamma]."""
    return [verify_greedy_seq(target[b], draft_tokens[b])
            for b in range(len(draft_tokens))]


def verify_sample(target, draft, draft_tokens, temperature, u_accept,
                  u_resample, seqs=None) -> list[SeqResult]:
    """target [B, gamma+1, V]; draft [B, gamma, V]; temperature [B] (<= 0:
    greedy sequence); u_accept [B, gamma]; u_resample [B].  ``seqs`` limits
    the work to a subset of sequence indices (results come back in that order).
    """
    idx = range(len(draft_tokens)) if seqs is None else seqs
    return [verify_sample_seq(target[b], draft[b], draft_tokens[b],
                              temperature[b], u_accept[b], u_resample[b])
            for b in idx]


def verify_sample_topkp(target, draft, draft_tokens, temperature, top_k, top_p,
                        u_accept, u_resample, seqs=None) -> list[SeqResult]:
    """Batch form of ``verify_sample_topkp_seq`` (same layout as verify_sample)."""
    idx = range(len(draft_tokens)) if seqs is None else seqs
    return [verify_sample_topkp_seq(target[b], draft[b], draft_tokens[b], temperature[b],
                                    top_k, top_p, u_accept[b], u_resample[b])
            for b in idx]


# ---------------------------------------------------------------------------
# several draft candidates per sequence ([MTP-blog] §6 进阶优化与扩展思路, item
# 2 多候选草稿: the target verifies n candidate drafts at once and the one with
# the longest accepted length is kept)
# ---------------------------------------------------------------------------
def verify_greedy_multi(target, draft_tokens) -> list[tuple[SeqResult, int]]:
    """target [B, n, gamma+1, V]: the target's rows for each candidate path;
    draft_tokens [B, n, gamma].  Each candidate is verified greedily on its
    own rows; the kept candidate is the one with the most accepted drafts, the
    lowest candidate index on ties.  Returns (its SeqResult, its index) per
    sequence."""
    out = []
    for b in range(len(draft_tokens)):
        res = [verify_greedy_seq(target[b][c], draft_tokens[b][c])
               for c in range(len(draft_tokens[b]))]
        best = 0
        for c in range(1, len(res)):
            if res[c].n > res[best].n:
                best = c
        out.append((res[best], best))
    return out


# ---------------------------------------------------------------------------
# fused lm_head: target logits = hidden @ W^T with the tied embedding
# ([MTP-deep] §3.1: lm_head shares embed_tokens; [Drafter] 高效 Embedder)
# ---------------------------------------------------------------------------
def lmhead_logits(hidden, W) -> np.ndarray:
    """l[r, x] = sum_k h[r, k] * W[x, k] in float64."""
    return _as_f64(hidden) @ _as_f64(W).T


def verify_lmhead_sample(hidden, W, draft, draft_tokens, temperature,
                         u_accept, u_resample, gamma, seqs=None):
    """Sampling verification where the target logits come from the lm_head.

    hidden [B*(gamma+1), H] holds, for sequence b, the hidden states of its
    gamma+1 verify positions in rows b*(gamma+1) .. b*(gamma+1)+gamma.
    """
    B = len(draft_tokens)
    idx = range(B) if seqs is None else seqs
    h = _as_f64(hidden)
    Wf = _as_f64(W)  # widened once for all sequences
    out = []
    for b in idx:
        rows = h[b * (gamma + 1):(b + 1) * (gamma + 1)]
        tp = lmhead_logits(rows, Wf)
        out.append(verify_sample_seq(tp, draft[b], draft_tokens[b],
                                     temperature[b], u_accept[b], u_resample[b]))
    return out
