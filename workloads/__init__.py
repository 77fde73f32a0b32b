"""Seeded synthetic inputs for the verify step (shared by tests and bench).

This module holds input recipes only: logits profiles, noise, temperatures,
draft tokens and uniforms.  It contains none of the verify arithmetic and
imports neither the oracle nor the CUDA library.

Recipes (the pages name no dataset; these stand in for the workloads they
describe):

* tiny      B=8,   gamma=4, V=4096,    fp32.  l_p ~ N(0, 2^2); l_q = l_p + N(0, 0.5^2).
* single    B=1,   gamma=4, V=262144,  bf16.  Zipf-shaped target: -1.1*log(rank)
            over a random permutation plus N(0, 0.3^2); l_q = l_p + N(0, sigma^2).
* batched   B=32,  gamma=4, V=262144,  bf16.  As ``single`` with sigma=0.5 and
            per-sequence T ~ U[0.5, 1.2].
* longdraft B=128, gamma=8, V=262144,  fp32.  Zipf target; per-sequence sigma ~
            U[0.1, 1.5]; even sequences greedy, odd ones sample at T=1.0.
* lmhead    hidden [64*5, 1536] ~ N(0,1) bf16; tied embedding W [262144, 1536] ~
            N(0, 0.02^2) bf16; l_q = bf16(h W^T + N(0, 0.5^2)); T=1.0.  The
            exact-sums variant puts h on a 1/8 grid and W on a 2^-11 grid so
            that h W^T is exact in fp32 in any summation order.

Draft tokens: a sampling sequence draws d_{j+1} from q_j = softmax(l_q[j]/T)
with the Gumbel-max trick; a greedy sequence (T <= 0) takes argmax l_q[j]
(the drafter's own greedy choice).  Uniforms are float32 in [0, 1), one per
draft position and one per sequence per round, from a Philox stream seeded
with the config seed (u_accept [R, B, gamma] first, then u_resample [R, B]).

bf16 arrays are returned as uint16 bit patterns (round to nearest even).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = ["VerifyInputs", "LmheadInputs", "CONFIGS", "make_round",
           "make_lmhead_round", "make_lmhead_W", "make_custom", "make_multi", "f32_to_bf16_bits",
           "bf16_bits_to_f32", "torch_round", "torch_lmhead_round", "CENTROID", "CentroidModel",
           "make_centroid_model", "make_centroid_round", "sample_sparse_drafts", "torch_centroid_model"]


# ---------------------------------------------------------------------------
# configurations
# ---------------------------------------------------------------------------
CONFIGS = {
    "tiny": dict(B=8, gamma=4, V=4096, dtype="f32", profile="normal",
                 target_sd=2.0, sigma=0.5, temperature=1.0, rounds=1000),
    "single": dict(B=1, gamma=4, V=262144, dtype="bf16", profile="zipf",
                   sigma=0.5, temperature=0.7, rounds=10000),
    "batched": dict(B=32, gamma=4, V=262144, dtype="bf16", profile="zipf",
                    sigma=0.5, temperature=("uniform", 0.5, 1.2), rounds=1000),
    "longdraft": dict(B=128, gamma=8, V=262144, dtype="f32", profile="zipf",
                      sigma=("uniform", 0.1, 1.5), temperature=("alternate", 0.0, 1.0),
                      rounds=1000),
    "lmhead": dict(B=64, gamma=4, V=262144, H=1536, dtype="bf16", sigma=0.5,
                   temperature=1.0, w_sd=0.02, rounds=1000),
}


@dataclass
class VerifyInputs:
    """One round of verify inputs (host arrays)."""

    B: int
    gamma: int
    V: int
    dtype: str               # "f32" or "bf16"
    target: np.ndarray       # [B, gamma+1, V] float32, or uint16 bf16 bits
    draft: np.ndarray        # [B, gamma, V] same dtype
    draft_tokens: np.ndarray  # int32 [B, gamma]
    temperature: np.ndarray  # float32 [B]; <= 0 means greedy
    u_accept: np.ndarray     # float32 [B, gamma]
    u_resample: np.ndarray   # float32 [B]


@dataclass
class LmheadInputs:
    B: int
    gamma: int
    V: int
    H: int
    hidden: np.ndarray       # uint16 bf16 bits [B*(gamma+1), H]
    W: np.ndarray            # uint16 bf16 bits [V, H]
    draft: np.ndarray        # uint16 bf16 bits [B, gamma, V]
    draft_tokens: np.ndarray
    temperature: np.ndarray
    u_accept: np.ndarray
    u_resample: np.ndarray


# ---------------------------------------------------------------------------
# bf16 helpers (storage format only)
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# numpy generators (canonical; identical on x86 and Arm)
# ---------------------------------------------------------------------------
def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, *stream])))


def _uniforms(seed: int, rounds: int, B: int, gamma: int, r: int):
    g = np.random.Generator(np.random.Philox(seed))
    ua = g.random((rounds, B, gamma), dtype=np.float32)
    ur = g.random((rounds, B), dtype=np.float32)
    return ua[r].copy(), ur[r].copy()


def _zipf_rows(rng: np.random.Generator, rows: int, V: int) -> np.ndarray:
    """-1.1*log(rank) over a random permutation per row, plus N(0, 0.3^2)."""
    base = (-1.1 * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    out = np.empty((rows, V), dtype=np.float32)
    for i in range(rows):
        out[i, rng.permutation(V)] = base
    out += rng.normal(0.0, 0.3, size=(rows, V)).astype(np.float32)
    return out


def _per_seq(spec, B: int, rng: np.random.Generator) -> np.ndarray:
    if isinstance(spec, tuple):
        kind, a, b = spec
        if kind == "uniform":
            return rng.uniform(a, b, size=B).astype(np.float32)
        if kind == "alternate":  # even sequences a, odd sequences b
            return np.where(np.arange(B) % 2 == 0, a, b).astype(np.float32)
        raise ValueError(kind)
    return np.full(B, spec, dtype=np.float32)


def _draft_tokens(rng, draft_f32: np.ndarray, temperature: np.ndarray) -> np.ndarray:
    """Sampling sequences: Gumbel-max over l_q/T; greedy ones: argmax l_q."""
    B, gamma, V = draft_f32.shape
    out = np.empty((B, gamma), dtype=np.int32)
    for b in range(B):
        T = float(temperature[b])
        if T > 0:
            g = rng.gumbel(size=(gamma, V))
            out[b] = np.argmax(draft_f32[b].astype(np.float64) / T + g, axis=1)
        else:
            out[b] = np.argmax(draft_f32[b], axis=1)
    return out


def make_custom(B: int, gamma: int, V: int, dtype: str = "f32", profile: str = "normal",
                target_sd: float = 2.0, sigma=0.5, temperature=1.0, seed: int = 0,
                r: int = 0, rounds: int = 1) -> VerifyInputs:
    """Build one round of inputs for an arbitrary shape with a config recipe."""
    rng = _rng(seed, 1, r)
    rows = B * (gamma + 1)
    if profile == "normal":
        tgt = rng.normal(0.0, target_sd, size=(rows, V)).astype(np.float32)
    elif profile == "zipf":
        tgt = _zipf_rows(rng, rows, V)
    else:
        raise ValueError(profile)
    tgt = tgt.reshape(B, gamma + 1, V)
    sig = _per_seq(sigma, B, rng)
    temp = _per_seq(temperature, B, rng)
    noise = rng.normal(0.0, 1.0, size=(B, gamma, V)).astype(np.float32)
    dft = tgt[:, :gamma, :] + noise * sig[:, None, None]
    if dtype == "bf16":
        tgt_s, dft_s = f32_to_bf16_bits(tgt), f32_to_bf16_bits(dft)
        dft_vals = bf16_bits_to_f32(dft_s)
    elif dtype == "f32":
        tgt_s, dft_s, dft_vals = tgt, dft.astype(np.float32), dft.astype(np.float32)
    else:
        raise ValueError(dtype)
    toks = _draft_tokens(_rng(seed, 2, r), dft_vals, temp)
    ua, ur = _uniforms(seed, rounds, B, gamma, r)
    return VerifyInputs(B, gamma, V, dtype, np.ascontiguousarray(tgt_s),
                        np.ascontiguousarray(dft_s), toks, temp, ua, ur)


def make_multi(B: int, n_cand: int, gamma: int = 4, V: int = 4096, dtype: str = "f32",
               profile: str = "normal", seed: int = 0, r: int = 0):
    """Several draft candidates per sequence: B*n_cand candidate paths drawn
    with ``make_custom`` (greedy drafts from draft logits with a per-path
    noise scale in [0.2, 1.5]), grouped [B, n_cand, ...].  Every candidate of
    a sequence starts from the same prefix, so their row 0 is made identical.
    Returns (target [B, n, gamma+1, V], draft_tokens [B, n, gamma])."""
    inp = make_custom(B * n_cand, gamma, V, dtype, profile, 2.0, ("uniform", 0.2, 1.5), 0.0,
                      seed, r, 1)
    tgt = inp.target.reshape(B, n_cand, gamma + 1, V).copy()
    tgt[:, 1:, 0, :] = tgt[:, :1, 0, :]
    toks = inp.draft_tokens.reshape(B, n_cand, gamma).copy()
    return tgt, toks


def make_round(config: str, r: int = 0, seed: int = 0, **overrides) -> VerifyInputs:
    """Round ``r`` of a named config (``tiny``, ``single``, ``batched``,
    ``longdraft``); keyword overrides replace recipe fields (e.g. sigma,
    temperature, B)."""
    c = dict(CONFIGS[config])
    c.update(overrides)
    return make_custom(c["B"], c["gamma"], c["V"], c["dtype"], c["profile"],
                       c.get("target_sd", 2.0), c["sigma"], c["temperature"],
                       seed, r, c["rounds"])


def make_lmhead_W(V: int = 262144, H: int = 1536, seed: int = 0,
                  exact_sums: bool = False) -> np.ndarray:
    """The tied embedding W [V, H] as bf16 bits (seed stream 3).

    exact_sums: W = k / 2048 with k = round(N(0, 0.02^2) * 2048) clipped to
    [-255, 255] (exact in bf16).  With hidden = k / 8, |k| <= 32, every
    product h*w is a multiple of 2^-14 and every partial sum of a logit is at
    most 1536 * 4 * 255/2048 < 2^10 in magnitude, so it is an integer
    multiple of 2^-14 below 2^24: exact in fp32 whatever the summation order.
    """
    c = CONFIGS["lmhead"]
    wr = _rng(seed, 3)
    w = wr.normal(0.0, c["w_sd"], size=(V, H)).astype(np.float32)
    if exact_sums:
        w = np.clip(np.rint(w * 2048.0), -255, 255).astype(np.float32) / np.float32(2048.0)
    return f32_to_bf16_bits(w)


def make_lmhead_round(r: int = 0, seed: int = 0, B: int = 64, gamma: int = 4,
                      V: int = 262144, H: int = 1536, W_bits: np.ndarray | None = None,
                      exact_sums: bool = False, temperature=None) -> LmheadInputs:
    """Round ``r`` of the fused lm_head recipe.  W is fixed across rounds
    (seed stream 3); pass ``W_bits`` (from ``make_lmhead_W`` with the same
    ``exact_sums``) to reuse one already generated.  ``exact_sums`` draws the
    hidden states on the 1/8 grid (see ``make_lmhead_W``); ``temperature``
    overrides the recipe's T (a scalar or a per-sequence spec)."""
    c = CONFIGS["lmhead"]
    if W_bits is None:
        W_bits = make_lmhead_W(V, H, seed, exact_sums)
    rng = _rng(seed, 4, r)
    R = B * (gamma + 1)
    h = rng.normal(0.0, 1.0, size=(R, H)).astype(np.float32)
    if exact_sums:
        h = np.clip(np.rint(h * 8.0), -32, 32).astype(np.float32) / np.float32(8.0)
    hid = f32_to_bf16_bits(h)
    # target logits (fp32) only to derive the draft logits; never an expected value
    tgt = bf16_bits_to_f32(hid) @ bf16_bits_to_f32(W_bits).T
    tgt = tgt.reshape(B, gamma + 1, V)[:, :gamma, :]
    dft = f32_to_bf16_bits(tgt + rng.normal(0.0, c["sigma"], size=tgt.shape).astype(np.float32))
    temp = _per_seq(c["temperature"] if temperature is None else temperature, B, rng)
    toks = _draft_tokens(_rng(seed, 5, r), bf16_bits_to_f32(dft), temp)
    ua, ur = _uniforms(seed, c["rounds"], B, gamma, r)
    return LmheadInputs(B, gamma, V, H, hid, W_bits, dft, toks, temp, ua, ur)


# ---------------------------------------------------------------------------
# torch generators (same recipes, drawn on the GPU; used for large bench pools)
# ---------------------------------------------------------------------------
def torch_round(config: str, r: int, device, seed: int = 0, **overrides) -> dict:
    """Same recipe as ``make_round`` but drawn with torch on ``device``.  The
    random stream differs from numpy's; nothing compares the two."""
    import torch

    c = dict(CONFIGS[config])
    c.update(overrides)
    B, gamma, V = c["B"], c["gamma"], c["V"]
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + r)
    rows = B * (gamma + 1)
    if c["profile"] == "zipf":
        base = -1.1 * torch.log(torch.arange(1, V + 1, device=device, dtype=torch.float32))
        keys = torch.rand(rows, V, generator=g, device=device)
        perm = torch.argsort(keys, dim=1)
        tgt = torch.empty(rows, V, device=device, dtype=torch.float32)
        tgt.scatter_(1, perm, base.expand(rows, V).contiguous())
        del keys, perm
        tgt += 0.3 * torch.randn(rows, V, generator=g, device=device)
    else:
        tgt = c.get("target_sd", 2.0) * torch.randn(rows, V, generator=g, device=device)
    tgt = tgt.view(B, gamma + 1, V)
    gcpu = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 9, r])))
    sig = torch.from_numpy(_per_seq(c["sigma"], B, gcpu)).to(device)
    temp = torch.from_numpy(_per_seq(c["temperature"], B, gcpu)).to(device)
    dft = tgt[:, :gamma, :] + sig.view(B, 1, 1) * torch.randn(B, gamma, V, generator=g, device=device)
    if c["dtype"] == "bf16":
        tgt, dft = tgt.to(torch.bfloat16), dft.to(torch.bfloat16)
    dvals = dft.float()
    u = torch.rand(B, gamma, V, generator=g, device=device).clamp_(min=1e-20)
    gum = -torch.log(-torch.log(u))
    del u
    tsafe = torch.where(temp > 0, temp, torch.ones_like(temp)).view(B, 1, 1)
    sampled = torch.argmax(dvals / tsafe + gum, dim=2)
    greedy = torch.argmax(dvals, dim=2)
    toks = torch.where((temp > 0).view(B, 1), sampled, greedy).to(torch.int32)
    del gum, dvals
    ua = torch.rand(B, gamma, generator=g, device=device)
    ur = torch.rand(B, generator=g, device=device)
    return dict(B=B, gamma=gamma, V=V, dtype=c["dtype"], target=tgt.contiguous(),
                draft=dft.contiguous(), draft_tokens=toks.contiguous(),
                temperature=temp.contiguous(), u_accept=ua.contiguous(),
                u_resample=ur.contiguous())


def torch_lmhead_round(r: int, device, W=None, seed: int = 0, B: int = 64,
                       gamma: int = 4, V: int = 262144, H: int = 1536) -> dict:
    """The lm_head recipe drawn with torch on ``device``."""
    import torch

    c = CONFIGS["lmhead"]
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + 77 + r)
    if W is None:
        gw = torch.Generator(device=device)
        gw.manual_seed(seed * 7919 + 3)
        W = (c["w_sd"] * torch.randn(V, H, generator=gw, device=device)).to(torch.bfloat16)
    R = B * (gamma + 1)
    hid = torch.randn(R, H, generator=g, device=device).to(torch.bfloat16)
    tgt = (hid.float() @ W.float().t()).view(B, gamma + 1, V)[:, :gamma, :]
    dft = (tgt + c["sigma"] * torch.randn(tgt.shape, generator=g, device=device)).to(torch.bfloat16)
    del tgt
    u = torch.rand(B, gamma, V, generator=g, device=device).clamp_(min=1e-20)
    toks = torch.argmax(dft.float() / c["temperature"] - torch.log(-torch.log(u)), dim=2).to(torch.int32)
    del u
    temp = torch.full((B,), c["temperature"], device=device)
    ua = torch.rand(B, gamma, generator=g, device=device)
    ur = torch.rand(B, generator=g, device=device)
    return dict(B=B, gamma=gamma, V=V, H=H, hidden=hid.contiguous(), W=W,
                draft=dft.contiguous(), draft_tokens=toks.contiguous(),
                temperature=temp, u_accept=ua.contiguous(), u_resample=ur.contiguous())


from .centroid import (CENTROID, CentroidModel, make_centroid_model,  # noqa: E402
                       make_centroid_round, sample_sparse_drafts, torch_centroid_model)
