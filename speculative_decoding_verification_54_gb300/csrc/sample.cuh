// sample.cuh — residual normaliser and inverse-CDF sampler.
//
// After a rejection at position n the token is drawn from
// w(x) = max(0, p_n(x) - q_n(x)) / Z ("Gemma 4 Multi-Token Prediction (MTP)
// 深度解析" §2.2; "自投机解码：层跳过与拒绝采样实现大模型推理加速" §3.2), and after a
// fully accepted draft from p_gamma (the bonus).  The draw is an inverse CDF
// in ascending vocabulary order: the smallest k with sum_{x<=k} w(x) > u*Z.
//
// Two levels keep it parallel:
//   residual_mass_kernel  one CTA per (sequence, chunk): the mass of w over the
//                         chunk (bonus masses come from the row partials);
//   sample_kernel         one warp per sequence: a scan over the chunk masses
//                         picks the chunk, a scan over that chunk's elements
//                         picks the token.
// Element weights are fp32; running sums across lanes and chunks are fp64,
// which on GB300 is kept to a few dozen operations per lane.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace specv {

constexpr int kMassThreads = 256;

struct SampleParams {
  const void* target;
  const void* draft;
  const float* u_resample;
  const float4* partials;
  const RowStat* rowstat;
  const SeqState* seq;
  float* mass;
  int32_t* out_tokens;
  int B, gamma, V, CE, cpr;
};

// Weight of one vocabulary entry of the selected row (pair), in the units of
// the chunk masses: residual -> max(0, p - q); bonus -> p * S (units of 2^mk).
struct WeightFn {
  float ks, mkp, mkq, invSp, invSq;
  bool residual;
  __device__ __forceinline__ float operator()(float xp, float xq) const {
    if (residual) {
      const float pp = ex2(fmaf(xp, ks, -mkp)) * invSp;
      const float qq = ex2(fmaf(xq, ks, -mkq)) * invSq;
      return fmaxf(0.f, pp - qq);
    }
    return ex2(fmaf(xp, ks, -mkp));
  }
};

__device__ __forceinline__ WeightFn make_weight(const SampleParams& p, int b, int n, int rowp,
                                                bool residual, float ks) {
  const int slots = 2 * p.gamma + 1;
  WeightFn f;
  f.ks = ks;
  f.residual = residual;
  const RowStat rp = p.rowstat[b * slots + rowp];
  f.mkp = rp.mk;
  f.invSp = ex2(-rp.lse2);
  if (residual) {
    const RowStat rq = p.rowstat[b * slots + p.gamma + 1 + n];
    f.mkq = rq.mk;
    f.invSq = ex2(-rq.lse2);
  } else {
    f.mkq = 0.f;
    f.invSq = 0.f;
  }
  return f;
}

template <typename T>
__device__ __forceinline__ const uint4* chunk_vec(const void* base, size_t row, int V, int c, int CE) {
  return reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(base) +
                                        (row * V + static_cast<size_t>(c) * CE) * sizeof(T));
}

// Warp-inclusive scan of one double per lane.
__device__ __forceinline__ double warp_scan_incl(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// ---------------------------------------------------------------------------
// K3: residual chunk masses
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kMassThreads) residual_mass_kernel(const SampleParams p) {
  __shared__ float warp_part[kMassThreads / 32];
  grid_dep_wait();
  const int b = blockIdx.y, c = blockIdx.x;
  const SeqState s = p.seq[b];
  if (s.mode != kModeResidual) return;
  constexpr int P = Elt<T>::kPerVec;
  const WeightFn f = make_weight(p, b, s.n, s.n, true, s.ks);
  const int g = p.gamma;
  const uint4* vp = chunk_vec<T>(p.target, static_cast<size_t>(b) * (g + 1) + s.n, p.V, c, p.CE);
  const uint4* vq = chunk_vec<T>(p.draft, static_cast<size_t>(b) * g + s.n, p.V, c, p.CE);
  const int len = min(p.CE, p.V - c * p.CE);
  const int nvec = len / P;
  float a0 = 0.f, a1 = 0.f;
  for (int i = threadIdx.x; i < nvec; i += kMassThreads) {
    float xp[P], xq[P], w[P];
    Elt<T>::unpack(vp[i], xp);
    Elt<T>::unpack(vq[i], xq);
#pragma unroll
    for (int j = 0; j < P; ++j) w[j] = f(xp[j], xq[j]);
    float t0 = 0.f, t1 = 0.f;
#pragma unroll
    for (int j = 0; j < P / 2; ++j) {
      t0 += w[j];
      t1 += w[P / 2 + j];
    }
    a0 += t0;
    a1 += t1;
  }
  float v = a0 + a1;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float sum = 0.f, cmp = 0.f;
    for (int w = 0; w < kMassThreads / 32; ++w) neumaier_add(sum, cmp, warp_part[w]);
    p.mass[static_cast<size_t>(b) * p.cpr + c] = sum + cmp;
  }
}

// ---------------------------------------------------------------------------
// K4: the inverse-CDF draw, one warp per sequence
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(32) sample_kernel(const SampleParams p) {
  grid_dep_wait();
  const int b = blockIdx.x, lane = threadIdx.x;
  const SeqState s = p.seq[b];
  if (s.mode != kModeResidual && s.mode != kModeBonus) return;
  const int g = p.gamma, slots = 2 * g + 1;
  float* mass = p.mass + static_cast<size_t>(b) * p.cpr;
  const int per = (p.cpr + 31) / 32;
  const int c0 = min(p.cpr, lane * per), c1 = min(p.cpr, c0 + per);

  bool residual = (s.mode == kModeResidual);
  const int rowp = residual ? s.n : g;

  // ---- level 1: which chunk (lane-contiguous chunk ranges) ----
  double lsum = 0.0;
  for (int c = c0; c < c1; ++c) lsum += static_cast<double>(mass[c]);
  double incl = warp_scan_incl(lsum);
  double Z = __shfl_sync(0xffffffffu, incl, 31);
  if (residual && !(Z > 0.0)) {
    // Z == 0 cannot happen in exact arithmetic; if rounding produces it, draw
    // from p_n itself (chunk masses from the row partials)
    const float4* P = p.partials + static_cast<size_t>(b * slots + s.n) * p.cpr;
    const float mk = p.rowstat[b * slots + s.n].mk;
    lsum = 0.0;
    for (int c = c0; c < c1; ++c) {
      const float4 q = P[c];
      mass[c] = q.y * ex2(q.w - mk);
      lsum += static_cast<double>(mass[c]);
    }
    incl = warp_scan_incl(lsum);
    Z = __shfl_sync(0xffffffffu, incl, 31);
    residual = false;  // weights of target row n as a plain row
  }
  const double target = static_cast<double>(p.u_resample[b]) * Z;
  const unsigned over = __ballot_sync(0xffffffffu, incl > target);
  int chunk = -1;
  double local = DBL_MAX;
  if (over) {
    const int L = __ffs(over) - 1;
    if (lane == L) {
      double run = incl - lsum;
      for (int c = c0; c < c1; ++c) {
        const double mc = static_cast<double>(mass[c]);
        if (run + mc > target) {
          chunk = c;
          local = target - run;
          break;
        }
        run += mc;
      }
      if (chunk < 0) {  // rounding inside the lane: its last nonzero chunk
        for (int c = c1 - 1; c >= c0; --c)
          if (mass[c] > 0.f) {
            chunk = c;
            break;
          }
      }
    }
    chunk = __shfl_sync(0xffffffffu, chunk, L);
    local = __shfl_sync(0xffffffffu, local, L);
  }
  if (chunk < 0) {  // u*Z at or beyond the total: the last nonzero chunk
    int last = -1;
    for (int c = c0; c < c1; ++c)
      if (mass[c] > 0.f) last = c;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
    chunk = last < 0 ? 0 : last;
    local = DBL_MAX;
  }

  // ---- level 2: which token inside the chunk (lane-contiguous vectors) ----
  const WeightFn f = make_weight(p, b, s.n, rowp, residual, s.ks);
  constexpr int P = Elt<T>::kPerVec;
  const uint4* vp = chunk_vec<T>(p.target, static_cast<size_t>(b) * (g + 1) + rowp, p.V, chunk, p.CE);
  const uint4* vq = residual ? chunk_vec<T>(p.draft, static_cast<size_t>(b) * g + s.n, p.V, chunk, p.CE)
                             : nullptr;
  const int len = min(p.CE, p.V - chunk * p.CE);
  const int nvec = len / P;
  const int vper = (nvec + 31) / 32;
  const int v0 = min(nvec, lane * vper), v1 = min(nvec, v0 + vper);
  float my = 0.f;
  int last_nz = -1;
  for (int i = v0; i < v1; ++i) {
    float xp[P], xq[P];
    Elt<T>::unpack(vp[i], xp);
    if (residual) Elt<T>::unpack(vq[i], xq);
    float t = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      const float w = f(xp[j], residual ? xq[j] : 0.f);
      t += w;
      if (w > 0.f) last_nz = i * P + j;
    }
    my += t;
  }
  const double cincl = warp_scan_incl(static_cast<double>(my));
  const unsigned cover = __ballot_sync(0xffffffffu, cincl > local);
  int tok = -1;
  if (cover) {
    const int L = __ffs(cover) - 1;
    if (lane == L) {
      double run = cincl - static_cast<double>(my);
      for (int i = v0; i < v1 && tok < 0; ++i) {
        float xp[P], xq[P];
        Elt<T>::unpack(vp[i], xp);
        if (residual) Elt<T>::unpack(vq[i], xq);
#pragma unroll
        for (int j = 0; j < P; ++j) {
          const float w = f(xp[j], residual ? xq[j] : 0.f);
          run += static_cast<double>(w);
          if (tok < 0 && run > local) tok = i * P + j;
        }
      }
      if (tok < 0) tok = last_nz;  // rounding inside the lane
    }
    tok = __shfl_sync(0xffffffffu, tok, L);
  }
  if (tok < 0) {  // beyond the chunk total: its last nonzero entry
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) last_nz = max(last_nz, __shfl_xor_sync(0xffffffffu, last_nz, off));
    tok = last_nz < 0 ? 0 : last_nz;
  }
  if (lane == 0) p.out_tokens[b * (g + 1) + s.n] = chunk * p.CE + tok;
}

}  // namespace specv
