"""Centroid-masked sparse draft head, and verification against its sparse q.

TEST INFRASTRUCTURE ONLY (see the package docstring): imported by ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs, never by the product
library, with which it shares no code.

[MTP-deep] §3.4 Centroids Masking and [Drafter] 高效 Embedder describe the
drafter head of the small Gemma 4 models.  The token embeddings are grouped
into clusters and stored cluster by cluster ("ordered embeddings": cluster c
owns the ordered rows cluster_off[c] .. cluster_off[c+1]-1, and ordered row i
is token ord2tok[i]).  One embedding per cluster (its centroid) scores the
clusters against the drafter's hidden state; the top_k clusters are kept, and
token logits (hidden . embedding) are computed only for the tokens of those
clusters, about top_k * V / n_clusters of them.  Tokens outside get no logit:
the draft distribution q is the softmax over the candidates and 0 elsewhere.

Readings where the pages are silent: the cluster score is the dot product with the
centroid (no bias, no scaling); the top_k are the largest scores with the
lowest cluster index first among equal scores; candidates are reported in
ascending token id.

Everything is float64.  bf16 inputs (uint16 bit patterns) widen exactly.
"""
from __future__ import annotations

import numpy as np

from .spec_oracle import _as_f64, _decide_and_draw, row_log_normaliser, verify_greedy_seq

__all__ = ["cluster_scores", "top_clusters", "centroid_head", "sparse_row_to_dense",
           "verify_sample_sparse"]


def cluster_scores(hidden, centroids) -> np.ndarray:
    """z[r, c] = hidden[r] . centroids[c] in float64 ([MTP-deep] §3.4 step 2:
    the hidden state predicts which clusters are most likely)."""
    return _as_f64(hidden) @ _as_f64(centroids).T


def top_clusters(scores_row, top_k: int) -> np.ndarray:
    """The top_k clusters of one row: largest score first, the lowest cluster
    index first among equal scores."""
    s = np.asarray(scores_row, dtype=np.float64)
    order = np.lexsort((np.arange(s.size), -s))  # by -score, then by index
    return order[:top_k]


def centroid_head(hidden, centroids, W_ord, cluster_off, ord2tok, top_k: int):
    """The sparse draft logits of every row of ``hidden`` [R, H].

    For row r: the top_k clusters by ``cluster_scores``; the candidates are
    the tokens of those clusters, each with logit hidden[r] . W_ord[i] for its
    ordered row i ([MTP-deep] §3.4 step 3; [Drafter] 高效 Embedder).  Returns a
    list of (tokens ascending as int64, logits float64) per row.
    """
    h = _as_f64(hidden)
    z = cluster_scores(h, centroids)
    off = np.asarray(cluster_off, dtype=np.int64)
    o2t = np.asarray(ord2tok, dtype=np.int64)
    out = []
    for r in range(h.shape[0]):
        sel = top_clusters(z[r], top_k)
        pos = np.concatenate([np.arange(off[c], off[c + 1]) for c in sel])
        logits = _as_f64(np.asarray(W_ord)[pos]) @ h[r]
        tok = o2t[pos]
        order = np.argsort(tok, kind="stable")
        out.append((tok[order], logits[order]))
    return out


def sparse_row_to_dense(tokens, logits, V: int) -> np.ndarray:
    """A draft logit row over the whole vocabulary: the candidates' logits,
    -inf elsewhere (so q = softmax over the candidates, 0 outside)."""
    row = np.full(V, -np.inf)
    row[np.asarray(tokens, dtype=np.int64)] = np.asarray(logits, dtype=np.float64)
    return row


def verify_sample_sparse(target, cand, draft_tokens, temperature, u_accept, u_resample,
                         seqs=None):
    """Rejection-sampling verification whose draft rows are sparse.

    target [B, gamma+1, V]; cand[b][j] = (tokens, logits) of draft row j of
    sequence b.  q_j is the softmax of the candidates' logits / T and 0 off the
    candidates (a row without candidates is q = 0 everywhere).  The rule is
    the dense one ([MTP-deep] §2.2; [Self-spec] §3.2): accept iff
    u < p(d)/q(d), q(d) = 0 accepting; after a rejection at n draw from
    max(0, p_n - q_n), which is p_n itself on every non-candidate token; after
    a full acceptance draw the bonus from p_gamma.
    """
    B = len(draft_tokens)
    idx = range(B) if seqs is None else seqs
    out = []
    for b in idx:
        T = float(temperature[b])
        if T <= 0.0:
            out.append(verify_greedy_seq(target[b], draft_tokens[b]))
            continue
        tp = _as_f64(target[b])
        V = tp.shape[-1]
        d = [int(x) for x in draft_tokens[b]]
        gamma = len(d)
        L_p = [row_log_normaliser(tp[j], T) for j in range(gamma + 1)]
        P = [np.exp(tp[j] / T - L_p[j]) for j in range(gamma + 1)]
        Q, L_q = [], []
        for (tok, lg) in cand[b]:
            if len(tok) == 0:
                Q.append(np.zeros(V))
                L_q.append(-np.inf)
                continue
            row = sparse_row_to_dense(tok, lg, V)
            L_q.append(row_log_normaliser(row, T))
            Q.append(np.exp(row / T - L_q[-1]))
        out.append(_decide_and_draw(P, Q, d, u_accept[b], u_resample[b], L_p, L_q))
    return out
