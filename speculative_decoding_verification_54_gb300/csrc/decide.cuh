// decide.cuh — row combine and per-sequence acceptance decision.
//
// Used by the tail kernel, whose CTAs each handle one sequence:
//   combine_row      one warp folds a row's chunk partials into (scaled max
//                    mk, log2 of the normaliser, argmax);
//   decide_sequence  one warp evaluates every draft position at once, one lane
//                    per position:
//     greedy   accept d_{j+1} iff d_{j+1} == argmax_j
//              ("自投机解码：层跳过与拒绝采样实现大模型推理加速" §3.1)
//     sampling accept iff u_accept[b,j] < p_j(d)/q_j(d)
//              ("Gemma 4 Multi-Token Prediction (MTP) 深度解析" §2.2)
//   and finds the first rejection n with a warp ballot.  Drafts before n are
//   emitted; position n gets the target argmax (greedy: the replacement, or
//   the bonus when n = gamma — "第 8 章 投机解码：一次前向，验证好几个字",
//   多出来的那一个 token 从哪来) or is left to the inverse-CDF draw.
//
// Arithmetic: GB300's FP64 rate is a small fraction of its FP32 rate, so the
// combine runs in fp32 with compensated (Neumaier) summation, and the ratio
// is formed as one exp2 of
//   (x_p - x_q)*ks - (mk_p - mk_q) - (log2 S_p - log2 S_q),
// three small differences, instead of a quotient of two rounded exps.  The
// rounding of mk = fl(M*ks) cancels because the same mk was subtracted from
// every exponent summed into S.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace specv {

constexpr int kCombineBatch = 8;  // partials each lane loads at once (256 per warp)

// Fold the cpr chunk partials {M, s, argmax, mk} of one row, warp-wide.
// Loads are issued in batches of 32*kBatch so that a few L2 round trips cover
// a row (kBatch = 8: one round trip for the 128 partials of a 262,144-entry
// bf16 row).  Lane 0's result is the one to use.
template <int kBatch = kCombineBatch>
__device__ __forceinline__ RowStat combine_row(const float4* P, int cpr, bool sampled) {
  constexpr int kCombineBatch = kBatch;
  const int lane = threadIdx.x & 31;
  float m = -FLT_MAX, mkmax = kNegHuge;
  int idx = -1;
  float s = 0.f, cmp = 0.f;
  float4 q[kCombineBatch];
  for (int base = 0; base < cpr; base += 32 * kCombineBatch) {
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) {
      const int c = base + lane + 32 * k;
      q[k] = (c < cpr) ? __ldcg(P + c) : make_float4(-FLT_MAX, 0.f, __int_as_float(-1), kNegHuge);
    }
    float bm = mkmax;
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) bm = fmaxf(bm, q[k].w);
    if (sampled) {
      const float sc = ex2(mkmax - bm);  // rescale the sum kept so far (it is 0 on the first batch)
      s *= sc;
      cmp *= sc;
#pragma unroll
      for (int k = 0; k < kCombineBatch; ++k) neumaier_add(s, cmp, q[k].y * ex2(q[k].w - bm));
    }
    mkmax = bm;
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) {
      const int qi = __float_as_int(q[k].z);
      if (q[k].x > m || (q[k].x == m && static_cast<unsigned>(qi) < static_cast<unsigned>(idx))) {
        m = q[k].x;
        idx = qi;
      }
    }
  }
  // lanes may hold different scaled maxima: rescale to the warp maximum
  float wm = mkmax;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, off));
  if (sampled) {
    const float sc = ex2(mkmax - wm);
    s *= sc;
    cmp *= sc;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, off);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
    if (om > m || (om == m && static_cast<unsigned>(oi) < static_cast<unsigned>(idx))) {
      m = om;
      idx = oi;
    }
    if (sampled) {
      const float os = __shfl_xor_sync(0xffffffffu, s, off);
      const float oc = __shfl_xor_sync(0xffffffffu, cmp, off);
      neumaier_add(s, cmp, os);
      cmp += oc;
    }
  }
  RowStat st;
  st.mk = wm;
  st.argmax = idx;
  st.pad = 0;
  st.lse2 = sampled ? log2f(s + cmp) : 0.f;
  return st;
}

struct DecideParams {
  const void* target;
  const void* draft;
  const int32_t* draft_tokens;
  const float* temperature;  // nullptr: greedy entry point
  const float* u_accept;
  int32_t* out_tokens;
  int32_t* out_num;
  float* out_debug;
  int* status;
  int gamma, V;
};

// What the decision reads from the call's inputs (not from the row reducer),
// one lane per draft position: loaded before the tail kernel waits for the
// reducer, so these loads overlap it.
struct DecideIn {
  int d;
  float xp, xq, u;
};

template <typename T>
__device__ __forceinline__ DecideIn prefetch_decide(const DecideParams& p, int b, bool greedy) {
  const int lane = threadIdx.x & 31;
  const int g = p.gamma;
  DecideIn in;
  in.d = -1;
  in.xp = in.xq = in.u = 0.f;
  if (lane < g) {
    in.d = p.draft_tokens[b * g + lane];
    if (!greedy && in.d >= 0 && in.d < p.V) {
      in.xp = Elt<T>::load1(p.target, (static_cast<size_t>(b) * (g + 1) + lane) * p.V + in.d);
      in.xq = Elt<T>::load1(p.draft, (static_cast<size_t>(b) * g + lane) * p.V + in.d);
      in.u = p.u_accept[b * g + lane];
    }
  }
  return in;
}

// Decide sequence b, warp-wide.  rs holds its combined rows (target rows
// 0..gamma, then draft rows 0..gamma-1); `in` the prefetched inputs.  Every
// CTA of the sequence computes the same decision; only the one with
// write_out stores the outputs.  The decision itself lands in *out (lane 0).
template <typename T>
__device__ __forceinline__ void decide_sequence(const DecideParams& p, int b, const RowStat* rs,
                                                const DecideIn& in, bool write_out, SeqState* out) {
  const int lane = threadIdx.x & 31;
  const int g = p.gamma;
  const bool greedy = (p.temperature == nullptr) || seq_is_greedy(p.temperature, b);
  const float ks = greedy ? 0.f : kLog2e / p.temperature[b];
  const int d = in.d;
  bool acc = false;
  float lp = 0.f, lq = 0.f;
  RowStat rp = {}, rq = {};
  if (lane <= g) rp = rs[lane];  // target row `lane`
  if (lane < g) {
    const bool valid = d >= 0 && d < p.V;
    if (!valid && write_out) atomicOr(p.status, kStatusBadToken);
    if (valid) {
      if (greedy) {
        acc = (d == rp.argmax);
      } else {
        rq = rs[g + 1 + lane];
        lp = fmaf(in.xp, ks, -rp.mk) - rp.lse2;  // log2 p(d), log2 q(d) (debug output)
        lq = fmaf(in.xq, ks, -rq.mk) - rq.lse2;
        // log2 of the ratio from three small differences (see header)
        const float t = (in.xp - in.xq) * ks - (rp.mk - rq.mk) - (rp.lse2 - rq.lse2);
        // q(d) == 0: the ratio is +inf and the draft is accepted
        const float rho = (in.xq == -INFINITY) ? INFINITY : ex2(t);
        acc = in.u < rho;
      }
    }
  }
  const unsigned mask = (1u << g) - 1u;
  const unsigned rej = ~__ballot_sync(0xffffffffu, acc) & mask;
  const int n = rej ? (__ffs(rej) - 1) : g;
  const int mode = greedy ? kModeGreedy : (n < g ? kModeResidual : kModeBonus);
  if (write_out && lane <= g) {
    int tok = -1;
    if (lane < n) tok = d;
    else if (lane == n && greedy) tok = rp.argmax;  // replacement or bonus
    p.out_tokens[b * (g + 1) + lane] = tok;
    if (p.out_debug != nullptr) {
      constexpr float kLn2 = 0.6931471805599453f;
      float4 dbg;
      if (greedy) {
        const float nan = __int_as_float(0x7fc00000);
        dbg = make_float4(nan, nan, nan, nan);
      } else if (lane < g) {
        dbg = make_float4(ex2(lp), ex2(lq), (rp.mk + rp.lse2) * kLn2, (rq.mk + rq.lse2) * kLn2);
      } else {
        dbg = make_float4(0.f, 0.f, (rp.mk + rp.lse2) * kLn2, 0.f);
      }
      reinterpret_cast<float4*>(p.out_debug)[b * (g + 1) + lane] = dbg;
    }
  }
  if (lane == 0) {
    if (write_out) p.out_num[b] = n;
    SeqState s;
    s.n = n;
    s.mode = mode;
    s.ks = ks;
    s.pad = 0;
    *out = s;
  }
}

// Several draft candidates per sequence ("Accelerating Gemma 4: faster
// inference with multi-token prediction drafters" §6, item 2 多候选草稿): each
// candidate was verified greedily as a sequence of its own (rows b*n + c);
// keep the one with the most accepted drafts, the lowest candidate index on
// ties.  One warp per sequence.
__global__ void __launch_bounds__(32) select_candidate_kernel(const int32_t* cand_tokens, const int32_t* cand_num,
                                                               int n_cand, int gamma, int32_t* out_tokens,
                                                               int32_t* out_num, int32_t* out_choice) {
  grid_dep_wait();
  const int b = blockIdx.x, lane = threadIdx.x;
  int best_n = -1, best_c = n_cand;
  for (int c = lane; c < n_cand; c += 32) {  // c grows within a lane: strict > keeps the lowest
    const int nn = cand_num[b * n_cand + c];
    if (nn > best_n) {
      best_n = nn;
      best_c = c;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const int on = __shfl_xor_sync(0xffffffffu, best_n, off);
    const int oc = __shfl_xor_sync(0xffffffffu, best_c, off);
    if (on > best_n || (on == best_n && oc < best_c)) {
      best_n = on;
      best_c = oc;
    }
  }
  const int32_t* src = cand_tokens + static_cast<size_t>(b * n_cand + best_c) * (gamma + 1);
  for (int j = lane; j <= gamma; j += 32) out_tokens[b * (gamma + 1) + j] = src[j];
  if (lane == 0) {
    out_num[b] = best_n;
    if (out_choice != nullptr) out_choice[b] = best_c;
  }
}

}  // namespace specv
