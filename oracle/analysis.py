"""Closed-form expectations for speculative decoding (fp64, CPU).

TEST INFRASTRUCTURE ONLY (same rules as ``spec_oracle``).

These are the analytic results the pages derive under the simplifying
assumption that every draft token is accepted independently with the same
probability alpha.  They pin the oracle's acceptance statistics and give the
host-side speed-up model.
"""
from __future__ import annotations

__all__ = ["expected_tokens_per_round", "speedup_naive", "speedup_layer_skip",
           "best_gamma"]


def expected_tokens_per_round(alpha: float, gamma: int) -> float:
    """E[len] = 1 + sum_{k=1..gamma} alpha^k = (1 - alpha^(gamma+1)) / (1 - alpha).

    At least one token per round: the corrected or bonus token.  From
    "自投机解码：层跳过与拒绝采样实现大模型推理加速" §4.1 and
    "第 8 章 投机解码：一次前向，验证好几个字" section 收益怎么算.
    """
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def speedup_naive(alpha: float, gamma: int, c: float) -> float:
    """S = E[len] / (1 + gamma*c): gamma draft passes of relative cost c plus one
    full verify pass ("自投机解码…" §4.2; "第 8 章 投机解码…" 收益怎么算, where
    1 + gamma*c is the cost factor 1.08 at gamma=4, c=0.02)."""
    return expected_tokens_per_round(alpha, gamma) / (1.0 + gamma * c)


def speedup_layer_skip(alpha: float, gamma: int, c: float) -> float:
    """S = E[len] / (1 - c + gamma*c): the layer-skip variant whose verify pass
    reuses the draft's shallow-layer KV cache and so costs about 1 - c
    ("自投机解码…" §4.2)."""
    return expected_tokens_per_round(alpha, gamma) / (1.0 - c + gamma * c)


def best_gamma(alpha: float, c: float, model=speedup_layer_skip,
               gammas=range(1, 33)) -> int:
    """The draft length that maximises the speed-up model ("自投机解码…" §4.2:
    maximise S over gamma)."""
    return max(gammas, key=lambda g: model(alpha, g, c))
