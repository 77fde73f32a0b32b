"""Host bookkeeping after a verify round (plain Python, CPU).

TEST INFRASTRUCTURE ONLY (same rules as ``spec_oracle``).

Per sequence the caller tracks seq_len (tokens: prompt + everything emitted),
kv_len (entries in the target's KV cache) and gamma (the draft length of the
next round).  Between rounds the newest token has no KV entry yet (it is the
first input of the next verify pass), so kv_len == seq_len - 1.

After a round in which n of gamma drafts were accepted:
* seq_len grows by n + 1: the accepted drafts and the replacement, resampled
  or bonus token ("第 8 章 投机解码：一次前向，验证好几个字", 多出来的那一个 token 从哪来);
* the verify pass appended gamma + 1 KV entries (the previous newest token and
  the gamma drafts); the entries after the accepted ones are dropped, so the
  cache keeps kv_len + n + 1 entries ("自投机解码：层跳过与拒绝采样实现大模型推理
  加速" §3.3: trim the KV cache to the accepted length and check each round
  that the cache length and the sequence length agree);
* gamma follows the heuristic schedule: +2 when every draft was accepted, -1
  when one was rejected ("Gemma 4 Multi-Token Prediction (MTP) 深度解析" §5.1),
  kept within [gamma_min, gamma_max] (the same page: beyond about 10 drafts the
  rejection rate rises and longer drafts stop paying).
"""
from __future__ import annotations

from dataclasses import dataclass

__all__ = ["RoundState", "round_update"]


@dataclass
class RoundState:
    gamma: int
    seq_len: int
    kv_len: int


def round_update(state: RoundState, n_accepted: int, gamma_min: int, gamma_max: int) -> int:
    """Apply one round to ``state`` in place.  Returns the number of KV
    entries to keep.  Raises ValueError when the bookkeeping is inconsistent
    (the cache and the sequence disagree before the round, or n is outside
    [0, gamma])."""
    g = state.gamma
    if state.kv_len != state.seq_len - 1:
        raise ValueError(f"kv_len {state.kv_len} != seq_len - 1 = {state.seq_len - 1}")
    if not 0 <= n_accepted <= g:
        raise ValueError(f"n_accepted {n_accepted} outside [0, {g}]")
    keep = state.kv_len + n_accepted + 1
    state.seq_len += n_accepted + 1
    state.kv_len = keep
    state.gamma = min(gamma_max, g + 2) if n_accepted == g else max(gamma_min, g - 1)
    return keep
