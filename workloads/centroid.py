"""Seeded synthetic inputs for the centroid-masked draft head and the sparse
verification that consumes its output.

Input recipes only: no verify arithmetic lives here.  The pages give the head's
shape (262,144 tokens, 2,048 clusters, top 32, about 4K candidates) but no
trained weights, so the clustering is synthetic.  Each token belongs to a
uniformly drawn cluster; a token's embedding is its cluster's centre plus
token noise, so a cluster's members are close; the centroid is the mean of the
members' (bf16) embeddings.  Target logits are the target hidden state times
the same embeddings; the drafter's hidden state is the target's plus noise.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import _rng, bf16_bits_to_f32, f32_to_bf16_bits

# Spreads chosen so that the drafter's candidates hold most of the target's
# mass and rounds both accept and reject (unstated on the pages).
CENTROID = dict(V=262144, H=1536, n_clusters=2048, top_k=32, mu_sd=0.05, eps_sd=0.004,
                draft_sd=0.05, temperature=0.7)


@dataclass
class CentroidModel:
    V: int
    H: int
    n_clusters: int
    W_ord: np.ndarray        # uint16 bf16 bits [V, H], cluster by cluster
    centroids: np.ndarray    # uint16 bf16 bits [n_clusters, H]
    cluster_off: np.ndarray  # int32 [n_clusters + 1]
    ord2tok: np.ndarray      # int32 [V]: token id of ordered row i
    tok2ord: np.ndarray      # int32 [V]: ordered row of token t


def _grid(x: np.ndarray, scale: float, lim: int) -> np.ndarray:
    """Round to multiples of 1/scale, clipped to +-lim/scale (exact in bf16 for lim <= 255)."""
    return (np.clip(np.rint(x * scale), -lim, lim) / scale).astype(np.float32)


def make_centroid_model(V: int = 4096, H: int = 64, n_clusters: int = 64, seed: int = 0,
                        exact_sums: bool = False, mu_sd: float | None = None,
                        eps_sd: float | None = None) -> CentroidModel:
    """Clustered embeddings (seed stream 7).

    exact_sums: embeddings and centroids are k/2048 with |k| <= 255 and hidden
    states k/8 with |k| <= 32 (``make_centroid_round``), so every dot product
    of length H <= 1536 is a sum of multiples of 2^-14 below 2^10: exact in
    fp32 in any order.
    """
    c = CENTROID
    mu_sd = c["mu_sd"] if mu_sd is None else mu_sd
    eps_sd = c["eps_sd"] if eps_sd is None else eps_sd
    rng = _rng(seed, 7)
    cl = rng.integers(0, n_clusters, size=V)
    ord2tok = np.lexsort((np.arange(V), cl)).astype(np.int32)  # by cluster, then token id
    counts = np.bincount(cl, minlength=n_clusters)
    off = np.zeros(n_clusters + 1, np.int32)
    off[1:] = np.cumsum(counts)
    tok2ord = np.empty(V, np.int32)
    tok2ord[ord2tok] = np.arange(V, dtype=np.int32)
    mu = rng.normal(0.0, mu_sd, size=(n_clusters, H)).astype(np.float32)
    w = mu[cl[ord2tok]] + rng.normal(0.0, eps_sd, size=(V, H)).astype(np.float32)
    if exact_sums:
        w = _grid(w, 2048.0, 255)
    W_bits = f32_to_bf16_bits(w)
    wf = bf16_bits_to_f32(W_bits).astype(np.float64)
    cen = mu.astype(np.float64).copy()
    nz = counts > 0
    sums = np.add.reduceat(wf, off[:-1][nz], axis=0) if nz.any() else np.zeros((0, H))
    cen[nz] = sums / counts[nz][:, None]
    cen = cen.astype(np.float32)
    if exact_sums:
        cen = _grid(cen, 2048.0, 255)
    return CentroidModel(V, H, n_clusters, W_bits, f32_to_bf16_bits(cen), off, ord2tok, tok2ord)


def make_centroid_round(model: CentroidModel, B: int, gamma: int, r: int = 0, seed: int = 0,
                        temperature=None, exact_sums: bool = False,
                        draft_sd: float | None = None) -> dict:
    """One round (seed stream 8): the target's hidden states [B*(gamma+1), H],
    target logits bf16(h . W) [B, gamma+1, V], the drafter's hidden states
    [B*gamma, H] (the target's at the same position plus N(0, draft_sd^2)),
    per-sequence temperature and the uniforms."""
    c = CENTROID
    draft_sd = c["draft_sd"] if draft_sd is None else draft_sd
    rng = _rng(seed, 8, r)
    H, V = model.H, model.V
    ht = rng.normal(0.0, 1.0, size=(B, gamma + 1, H)).astype(np.float32)
    hd = ht[:, :gamma] + rng.normal(0.0, draft_sd, size=(B, gamma, H)).astype(np.float32)
    if exact_sums:
        ht, hd = _grid(ht, 8.0, 32), _grid(hd, 8.0, 32)
    ht_bits, hd_bits = f32_to_bf16_bits(ht), f32_to_bf16_bits(hd)
    w_tok = bf16_bits_to_f32(model.W_ord[model.tok2ord])  # token order
    logits = bf16_bits_to_f32(ht_bits).reshape(-1, H) @ w_tok.T
    target = f32_to_bf16_bits(logits.astype(np.float32)).reshape(B, gamma + 1, V)
    T = c["temperature"] if temperature is None else temperature
    temp = np.full(B, T, np.float32) if np.isscalar(T) else np.asarray(T, np.float32)
    ua = rng.random((B, gamma), dtype=np.float32)
    ur = rng.random(B, dtype=np.float32)
    return dict(B=B, gamma=gamma, V=V, H=H, hidden_target=ht_bits.reshape(-1, H),
                hidden_draft=hd_bits.reshape(-1, H), target=target, temperature=temp,
                u_accept=ua, u_resample=ur)


def sample_sparse_drafts(cand, temperature, gamma: int, seed: int = 0, r: int = 0) -> np.ndarray:
    """Draft tokens drawn from sparse draft rows (seed stream 9): cand[b*gamma + j]
    = (tokens, logits); a sampling sequence takes the Gumbel-max over its
    candidates' logits / T, a greedy one (T <= 0) the largest logit (lowest
    token on ties)."""
    rng = _rng(seed, 9, r)
    B = len(temperature)
    out = np.zeros((B, gamma), np.int32)
    for b in range(B):
        T = float(temperature[b])
        for j in range(gamma):
            tok, lg = cand[b * gamma + j]
            lg = np.asarray(lg, np.float64)
            if T > 0:
                g = -np.log(-np.log(np.clip(rng.random(lg.size), 1e-300, 1.0)))
                out[b, j] = tok[int(np.argmax(lg / T + g))]
            else:
                out[b, j] = tok[int(np.argmax(lg))]
    return out


def torch_centroid_model(device, V: int | None = None, H: int | None = None, n_clusters: int | None = None,
                         seed: int = 0) -> dict:
    """The clustered-embedding recipe drawn with torch on ``device`` (a
    different random stream from ``make_centroid_model``): W_ord [V, H] bf16,
    centroids [n_clusters, H] bf16, cluster_off int32 [n_clusters+1], ord2tok
    int32 [V]."""
    import torch

    c = CENTROID
    V = c["V"] if V is None else V
    H = c["H"] if H is None else H
    n_clusters = c["n_clusters"] if n_clusters is None else n_clusters
    g = torch.Generator(device=device)
    g.manual_seed(seed * 7919 + 17)
    cl = torch.randint(0, n_clusters, (V,), generator=g, device=device)
    ord2tok = torch.argsort(cl.to(torch.int64) * V + torch.arange(V, device=device))
    counts = torch.bincount(cl, minlength=n_clusters)
    off = torch.zeros(n_clusters + 1, dtype=torch.int32, device=device)
    off[1:] = torch.cumsum(counts, 0).to(torch.int32)
    mu = c["mu_sd"] * torch.randn(n_clusters, H, generator=g, device=device)
    cl_ord = cl[ord2tok]
    w = (mu[cl_ord] + c["eps_sd"] * torch.randn(V, H, generator=g, device=device)).to(torch.bfloat16)
    sums = torch.zeros(n_clusters, H, device=device).index_add_(0, cl_ord, w.float())
    cen = torch.where(counts[:, None] > 0, sums / counts.clamp(min=1)[:, None], mu).to(torch.bfloat16)
    return dict(V=V, H=H, n_clusters=n_clusters, W_ord=w.contiguous(), centroids=cen.contiguous(),
                cluster_off=off, ord2tok=ord2tok.to(torch.int32).contiguous())
