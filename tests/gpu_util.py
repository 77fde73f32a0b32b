"""Helpers for the GPU parity tests: run the C ABI on host inputs and compare
its output with the fp64 oracle under the agreed tolerance.

Tolerance (from the stated target): greedy counts and tokens bit-exact;
sampling decisions and tokens exact unless a uniform lies within 1e-6 of the
acceptance or CDF boundary it was compared with (such cases are counted and
reported, not failed); probabilities within 1e-5 absolute.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BOUNDARY_WINDOW = 1e-6
PROB_ATOL = 1e-5


def to_device(inp, dev):
    import torch

    def logits(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    return dict(
        target=logits(inp.target), draft=logits(inp.draft),
        draft_tokens=torch.from_numpy(np.ascontiguousarray(inp.draft_tokens)).to(dev),
        temperature=torch.from_numpy(np.ascontiguousarray(inp.temperature)).to(dev),
        u_accept=torch.from_numpy(np.ascontiguousarray(inp.u_accept)).to(dev),
        u_resample=torch.from_numpy(np.ascontiguousarray(inp.u_resample)).to(dev))


def run_sample(sv, d, ws, debug=True):
    import torch
    B, g1, V = d["target"].shape
    out = torch.full((B, g1), -7, dtype=torch.int32, device=d["target"].device)
    num = torch.full((B,), -7, dtype=torch.int32, device=d["target"].device)
    dbg = torch.zeros((B, g1, 4), dtype=torch.float32, device=d["target"].device) if debug else None
    sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["temperature"],
                          d["u_accept"], d["u_resample"], out, num, ws, out_debug=dbg)
    st = sv.spec_verify_status(ws)
    return out.cpu().numpy(), num.cpu().numpy(), (dbg.cpu().numpy() if debug else None), st


def run_greedy(sv, d, ws):
    import torch
    B, g1, V = d["target"].shape
    out = torch.full((B, g1), -7, dtype=torch.int32, device=d["target"].device)
    num = torch.full((B,), -7, dtype=torch.int32, device=d["target"].device)
    sv.spec_verify_greedy(d["target"], d["draft_tokens"], out, num, ws)
    st = sv.spec_verify_status(ws)
    return out.cpu().numpy(), num.cpu().numpy(), st


@dataclass
class Tally:
    checked: int = 0
    exact: int = 0
    excused: int = 0
    failures: list = field(default_factory=list)
    max_prob_err: float = 0.0

    def merge(self, o):
        self.checked += o.checked
        self.exact += o.exact
        self.excused += o.excused
        self.failures += o.failures
        self.max_prob_err = max(self.max_prob_err, o.max_prob_err)
        return self


def compare(ref, tokens, num, dbg=None, seqs=None, label=""):
    """Compare oracle SeqResults with the GPU outputs (rows ``seqs``)."""
    t = Tally()
    idx = list(range(len(ref))) if seqs is None else list(seqs)
    for r, b in zip(ref, idx):
        t.checked += 1
        same = int(num[b]) == r.n and [int(x) for x in tokens[b]] == r.tokens
        if same:
            t.exact += 1
        elif r.margin < BOUNDARY_WINDOW:
            t.excused += 1
        else:
            t.failures.append((label, b, r.n, r.tokens, int(num[b]), [int(x) for x in tokens[b]],
                               r.margin, r.path))
        if dbg is not None and r.path != "greedy":
            g = len(r.p_tok)
            for j in range(g):
                t.max_prob_err = max(t.max_prob_err, abs(dbg[b, j, 0] - r.p_tok[j]),
                                     abs(dbg[b, j, 1] - r.q_tok[j]))
                for k, L in ((2, r.L_p[j]), (3, r.L_q[j])):
                    rel = abs(dbg[b, j, k] - L) / max(1.0, abs(L))
                    if rel > 1e-5:
                        t.failures.append((label, b, "L", j, k, float(dbg[b, j, k]), L))
            relg = abs(dbg[b, g, 2] - r.L_p[g]) / max(1.0, abs(r.L_p[g]))
            if relg > 1e-5:
                t.failures.append((label, b, "Lgamma", float(dbg[b, g, 2]), r.L_p[g]))
    return t


def assert_tally(t: Tally, max_excused_frac=0.01):
    assert not t.failures, f"{len(t.failures)} unexcused mismatches, first: {t.failures[:3]}"
    assert t.max_prob_err <= PROB_ATOL, t.max_prob_err
    assert t.excused <= max(2, max_excused_frac * t.checked), (t.excused, t.checked)
