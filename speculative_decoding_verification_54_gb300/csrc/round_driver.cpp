// round_driver.cpp — host bookkeeping after a verify round (no GPU work).
//
// Per sequence the caller keeps seq_len (prompt + emitted tokens), kv_len
// (entries in the target's KV cache) and gamma (the next round's draft
// length).  Between rounds the newest token has no KV entry yet, so
// kv_len == seq_len - 1.  After a round with n of gamma drafts accepted:
//   * seq_len += n + 1: the accepted drafts and the replacement / resampled /
//     bonus token ("第 8 章 投机解码：一次前向，验证好几个字", 多出来的那一个 token
//     从哪来);
//   * the verify pass appended gamma + 1 KV entries (the previous newest token
//     and the drafts); the cache keeps kv_len + n + 1 of them and drops the
//     rest ("自投机解码：层跳过与拒绝采样实现大模型推理加速" §3.3: trim to the
//     accepted length, and check every round that cache length and sequence
//     length agree);
//   * gamma += 2 when every draft was accepted, gamma -= 1 otherwise, kept in
//     [gamma_min, gamma_max] ("Gemma 4 Multi-Token Prediction (MTP) 深度解析"
//     §5.1, the heuristic schedule).
#include <cstdint>

#include "spec_verify.h"

extern "C" int spec_round_update(spec_round_state* states, const int32_t* num_accepted, int B, int gamma_min,
                                 int gamma_max, int64_t* kv_keep, int* first_bad) {
  if (first_bad != nullptr) *first_bad = -1;
  if (states == nullptr || num_accepted == nullptr || B < 0) return SPEC_ERR_INVALID_ARG;
  if (gamma_min < 1 || gamma_max > SPEC_MAX_GAMMA || gamma_min > gamma_max) return SPEC_ERR_INVALID_ARG;
  // validate every sequence first: nothing changes unless all are consistent
  for (int b = 0; b < B; ++b) {
    const spec_round_state& s = states[b];
    const int32_t n = num_accepted[b];
    if (s.gamma < 1 || s.seq_len < 1 || s.kv_len != s.seq_len - 1 || n < 0 || n > s.gamma) {
      if (first_bad != nullptr) *first_bad = b;
      return SPEC_ERR_STATE;
    }
  }
  for (int b = 0; b < B; ++b) {
    spec_round_state& s = states[b];
    const int32_t n = num_accepted[b];
    const int64_t keep = s.kv_len + n + 1;
    s.seq_len += n + 1;
    s.kv_len = keep;
    if (kv_keep != nullptr) kv_keep[b] = keep;
    const int32_t g = (n == s.gamma) ? s.gamma + 2 : s.gamma - 1;
    s.gamma = g < gamma_min ? gamma_min : (g > gamma_max ? gamma_max : g);
  }
  return SPEC_OK;
}
