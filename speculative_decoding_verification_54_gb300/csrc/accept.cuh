// accept.cuh — per-sequence acceptance evaluator.
//
// One CTA per sequence.  Its warps first combine the chunk partials of each
// row into (scaled max mk, log2 of the normaliser, argmax).  Warp 0 then
// evaluates every draft position at once, one lane per position:
//   greedy   accept d_{j+1} iff d_{j+1} == argmax_j
//            ("自投机解码：层跳过与拒绝采样实现大模型推理加速" §3.1)
//   sampling accept iff u_accept[b,j] < p_j(d)/q_j(d)
//            ("Gemma 4 Multi-Token Prediction (MTP) 深度解析" §2.2)
// and finds the first rejection n with a warp ballot.  Drafts before n are
// emitted; position n gets the target argmax (greedy) or is left for the
// residual sampler.  When a sampling sequence accepts everything, the chunk
// masses of p_gamma are formed here from the partials, so the bonus draw
// ("第 8 章 投机解码：一次前向，验证好几个字", 多出来的那一个 token 从哪来) needs no second
// pass over the row.
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

constexpr int kAcceptThreads = 256;

struct AcceptParams {
  const void* target;
  const void* draft;
  const int32_t* draft_tokens;
  const float* temperature;  // nullptr: greedy entry point
  const float* u_accept;
  const float4* partials;
  RowStat* rowstat;  // [B*(2*gamma+1)]
  SeqState* seq;     // [B]
  float* mass;       // [B*cpr] chunk masses for the final draw
  int32_t* out_tokens;
  int32_t* out_num;
  float* out_debug;
  int* status;
  int B, gamma, V, CE, cpr;
};

template <typename T>
__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(const AcceptParams p) {
  __shared__ RowStat rs[2 * 31 + 1];
  __shared__ int s_mode;
  grid_dep_wait();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.gamma, slots = 2 * g + 1;
  const bool greedy = (p.temperature == nullptr) || seq_is_greedy(p.temperature, b);
  const float ks = greedy ? 0.f : kLog2e / p.temperature[b];
  const int nrows = greedy ? g + 1 : 2 * g + 1;

  // ---- combine chunk partials per row -------------------------------------
  for (int r = warp; r < nrows; r += kAcceptThreads / 32) {
    const float4* P = p.partials + static_cast<size_t>(b * slots + r) * p.cpr;
    float m = -FLT_MAX, mkmax = kNegHuge;
    int idx = -1;
    for (int c = lane; c < p.cpr; c += 32) {
      const float4 q = P[c];
      const int qi = __float_as_int(q.z);
      if (q.x > m || (q.x == m && static_cast<unsigned>(qi) < static_cast<unsigned>(idx))) {
        m = q.x;
        idx = qi;
      }
      mkmax = fmaxf(mkmax, q.w);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, off);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
      if (om > m || (om == m && static_cast<unsigned>(oi) < static_cast<unsigned>(idx))) {
        m = om;
        idx = oi;
      }
      mkmax = fmaxf(mkmax, __shfl_xor_sync(0xffffffffu, mkmax, off));
    }
    float S = 0.f;
    if (!greedy) {
      float s = 0.f, cmp = 0.f;
      for (int c = lane; c < p.cpr; c += 32) {
        const float4 q = P[c];
        neumaier_add(s, cmp, q.y * ex2(q.w - mkmax));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, s, off);
        const float oc = __shfl_xor_sync(0xffffffffu, cmp, off);
        neumaier_add(s, cmp, os);
        cmp += oc;
      }
      S = s + cmp;
    }
    if (lane == 0) {
      RowStat st;
      st.mk = mkmax;
      st.argmax = idx;
      st.lse2 = greedy ? 0.f : log2f(S);
      st.pad = 0;
      rs[r] = st;
      p.rowstat[b * slots + r] = st;
    }
  }
  __syncthreads();

  // ---- decisions: one lane per draft position -----------------------------
  if (warp == 0) {
    int d = -1;
    bool acc = false;
    float lp = 0.f, lq = 0.f;
    if (lane < g) {
      d = p.draft_tokens[b * g + lane];
      const bool valid = d >= 0 && d < p.V;
      if (!valid) atomicOr(p.status, kStatusBadToken);
      if (valid) {
        if (greedy) {
          acc = (d == rs[lane].argmax);
        } else {
          const float xp = Elt<T>::load1(p.target, (static_cast<size_t>(b) * (g + 1) + lane) * p.V + d);
          const float xq = Elt<T>::load1(p.draft, (static_cast<size_t>(b) * g + lane) * p.V + d);
          const RowStat rp = rs[lane], rq = rs[g + 1 + lane];
          // log2 p(d) and log2 q(d), for the debug output
          lp = (fmaf(xp, ks, -rp.mk)) - rp.lse2;
          lq = (fmaf(xq, ks, -rq.mk)) - rq.lse2;
          // log2 of the ratio from three small differences (see header)
          const float t = (xp - xq) * ks - (rp.mk - rq.mk) - (rp.lse2 - rq.lse2);
          // q(d) == 0: the ratio is +inf and the draft is accepted
          const float rho = (xq == -INFINITY) ? INFINITY : ex2(t);
          acc = p.u_accept[b * g + lane] < rho;
        }
      }
    }
    const unsigned mask = (1u << g) - 1u;
    const unsigned rej = ~__ballot_sync(0xffffffffu, acc) & mask;
    const int n = rej ? (__ffs(rej) - 1) : g;
    const int mode = greedy ? kModeGreedy : (n < g ? kModeResidual : kModeBonus);
    if (lane <= g) {
      int tok = -1;
      if (lane < n) tok = d;
      else if (lane == n && greedy) tok = rs[n].argmax;
      p.out_tokens[b * (g + 1) + lane] = tok;
      if (p.out_debug != nullptr) {
        constexpr float kLn2 = 0.6931471805599453f;
        float4 dbg;
        if (greedy) {
          const float nan = __int_as_float(0x7fc00000);
          dbg = make_float4(nan, nan, nan, nan);
        } else if (lane < g) {
          const RowStat rp = rs[lane], rq = rs[g + 1 + lane];
          dbg = make_float4(ex2(lp), ex2(lq), (rp.mk + rp.lse2) * kLn2, (rq.mk + rq.lse2) * kLn2);
        } else {
          const RowStat rp = rs[g];
          dbg = make_float4(0.f, 0.f, (rp.mk + rp.lse2) * kLn2, 0.f);
        }
        reinterpret_cast<float4*>(p.out_debug)[b * (g + 1) + lane] = dbg;
      }
    }
    if (lane == 0) {
      p.out_num[b] = n;
      SeqState s;
      s.n = n;
      s.mode = mode;
      s.ks = ks;
      s.pad = 0;
      p.seq[b] = s;
      s_mode = mode;
    }
  }
  __syncthreads();

  // ---- bonus: chunk masses of p_gamma straight from the partials ----------
  if (s_mode == kModeBonus) {
    const float4* P = p.partials + static_cast<size_t>(b * slots + g) * p.cpr;
    const float mk = rs[g].mk;
    for (int c = threadIdx.x; c < p.cpr; c += kAcceptThreads) {
      const float4 q = P[c];
      p.mass[static_cast<size_t>(b) * p.cpr + c] = q.y * ex2(q.w - mk);
    }
  }
}

}  // namespace specv
