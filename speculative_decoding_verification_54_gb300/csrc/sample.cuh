// sample.cuh — residual normaliser and inverse-CDF sampler.
//
// After a rejection at position n the token is drawn from
// w(x) = max(0, p_n(x) - q_n(x)) / Z ("Gemma 4 Multi-Token Prediction (MTP)
// 深度解析" §2.2; "自投机解码：层跳过与拒绝采样实现大模型推理加速" §3.2), and after a
// fully accepted draft from p_gamma (the bonus).  The draw is an inverse CDF
// in ascending vocabulary order: the smallest k with sum_{x<=k} w(x) > u*Z.
//
// Two levels keep it parallel:
//   residual_mass_kernel  one CTA per (sequence, chunk): the fp64 mass of w over
//                         the chunk (bonus masses come from the row partials);
//   sample_kernel         one CTA per sequence: an fp64 block scan over the
//                         chunk masses picks the chunk, then a block scan over
//                         that chunk's elements picks the token.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace specv {

constexpr int kSampleThreads = 256;

struct SampleParams {
  const void* target;
  const void* draft;
  const float* u_resample;
  const float4* partials;
  const RowStat* rowstat;
  const SeqState* seq;
  double* mass;
  int32_t* out_tokens;
  int B, gamma, V, CE, cpr;
};

// Per-element weight of the chosen row (pair), in the same units as the chunk
// masses: residual -> max(0, p - q) in probability units; bonus -> p * 2^L in
// units of 2^mk.
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

__device__ __forceinline__ WeightFn make_weight(const SampleParams& p, int b, const SeqState& s) {
  const int slots = 2 * p.gamma + 1;
  WeightFn f;
  f.ks = s.ks;
  f.residual = (s.mode == kModeResidual);
  const int rowp = f.residual ? s.n : p.gamma;
  const RowStat rp = p.rowstat[b * slots + rowp];
  f.mkp = rp.mk;
  f.invSp = static_cast<float>(exp2(-rp.lse2));
  if (f.residual) {
    const RowStat rq = p.rowstat[b * slots + p.gamma + 1 + s.n];
    f.mkq = rq.mk;
    f.invSq = static_cast<float>(exp2(-rq.lse2));
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

// Block-wide inclusive scan of one double per thread.  Returns the inclusive
// value; *total gets the block total.
__device__ __forceinline__ double block_inclusive_scan(double v, double* total) {
  __shared__ double warp_tot[kSampleThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  double before = 0.0, tot = 0.0;
  for (int w = 0; w < kSampleThreads / 32; ++w) {
    if (w < warp) before += warp_tot[w];
    tot += warp_tot[w];
  }
  __syncthreads();
  *total = tot;
  return v + before;
}

__device__ __forceinline__ int block_max_int(int v) {
  __shared__ int red[kSampleThreads / 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  int r = red[0];
  for (int w = 1; w < kSampleThreads / 32; ++w) r = max(r, red[w]);
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------------------
// K3: residual chunk masses
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kSampleThreads) residual_mass_kernel(const SampleParams p) {
  grid_dep_wait();
  const int b = blockIdx.y, c = blockIdx.x;
  const SeqState s = p.seq[b];
  if (s.mode != kModeResidual) return;
  constexpr int P = Elt<T>::kPerVec;
  const WeightFn f = make_weight(p, b, s);
  const int g = p.gamma;
  const uint4* vp = chunk_vec<T>(p.target, static_cast<size_t>(b) * (g + 1) + s.n, p.V, c, p.CE);
  const uint4* vq = chunk_vec<T>(p.draft, static_cast<size_t>(b) * g + s.n, p.V, c, p.CE);
  const int len = min(p.CE, p.V - c * p.CE);
  const int nvec = len / P;
  float a0 = 0.f, a1 = 0.f;
  for (int i = threadIdx.x; i < nvec; i += kSampleThreads) {
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
  double v = static_cast<double>(a0) + static_cast<double>(a1);
  double tot;
  block_inclusive_scan(v, &tot);
  if (threadIdx.x == 0) p.mass[static_cast<size_t>(b) * p.cpr + c] = tot;
}

// ---------------------------------------------------------------------------
// K4: the inverse-CDF draw
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const SampleParams p) {
  __shared__ int s_chunk;
  __shared__ double s_local;
  __shared__ int s_tok;
  grid_dep_wait();
  const int b = blockIdx.x;
  SeqState s = p.seq[b];
  if (s.mode != kModeResidual && s.mode != kModeBonus) return;
  const int g = p.gamma, slots = 2 * g + 1;
  double* mass = p.mass + static_cast<size_t>(b) * p.cpr;
  const int per = (p.cpr + kSampleThreads - 1) / kSampleThreads;
  const int c0 = min(p.cpr, static_cast<int>(threadIdx.x) * per), c1 = min(p.cpr, c0 + per);

  // ---- level 1: which chunk ----
  double tsum = 0.0;
  for (int c = c0; c < c1; ++c) tsum += mass[c];
  double Z;
  double incl = block_inclusive_scan(tsum, &Z);
  bool residual = (s.mode == kModeResidual);
  int rowp = residual ? s.n : g;
  if (residual && !(Z > 0.0)) {
    // Z == 0 cannot happen in exact arithmetic; if rounding produces it, draw
    // from p_n itself (chunk masses from the row partials)
    const float4* P = p.partials + static_cast<size_t>(b * slots + s.n) * p.cpr;
    const double mk = static_cast<double>(p.rowstat[b * slots + s.n].mk);
    tsum = 0.0;
    for (int c = c0; c < c1; ++c) {
      const float4 q = P[c];
      mass[c] = static_cast<double>(q.y) * exp2(static_cast<double>(q.w) - mk);
      tsum += mass[c];
    }
    incl = block_inclusive_scan(tsum, &Z);
    residual = false;  // weights of row n as a plain target row
  }
  const double target = static_cast<double>(p.u_resample[b]) * Z;
  if (threadIdx.x == 0) s_chunk = -1;
  __syncthreads();
  const double excl = incl - tsum;
  if (excl <= target && incl > target) {
    double run = excl;
    for (int c = c0; c < c1; ++c) {
      if (run + mass[c] > target) {
        s_chunk = c;
        s_local = target - run;
        break;
      }
      run += mass[c];
    }
  }
  __syncthreads();
  int chunk = s_chunk;
  double local = s_local;
  if (chunk < 0) {  // rounding left no chunk above u*Z: take the last nonzero one
    int last = -1;
    for (int c = c0; c < c1; ++c)
      if (mass[c] > 0.0) last = c;
    chunk = block_max_int(last);
    local = DBL_MAX;
    if (chunk < 0) chunk = 0;
  }

  // ---- level 2: which token inside the chunk ----
  WeightFn f;
  {
    const RowStat rp = p.rowstat[b * slots + rowp];
    f.ks = s.ks;
    f.residual = residual;
    f.mkp = rp.mk;
    f.invSp = static_cast<float>(exp2(-rp.lse2));
    if (residual) {
      const RowStat rq = p.rowstat[b * slots + g + 1 + s.n];
      f.mkq = rq.mk;
      f.invSq = static_cast<float>(exp2(-rq.lse2));
    } else {
      f.mkq = 0.f;
      f.invSq = 0.f;
    }
  }
  constexpr int P = Elt<T>::kPerVec;
  const uint4* vp = chunk_vec<T>(p.target, static_cast<size_t>(b) * (g + 1) + rowp, p.V, chunk, p.CE);
  const uint4* vq = residual ? chunk_vec<T>(p.draft, static_cast<size_t>(b) * g + s.n, p.V, chunk, p.CE)
                             : nullptr;
  const int len = min(p.CE, p.V - chunk * p.CE);
  const int nvec = len / P;
  const int vper = (nvec + kSampleThreads - 1) / kSampleThreads;
  const int v0 = min(nvec, static_cast<int>(threadIdx.x) * vper), v1 = min(nvec, v0 + vper);
  double my = 0.0;
  int last_nz = -1;
  for (int i = v0; i < v1; ++i) {
    float xp[P], xq[P];
    Elt<T>::unpack(vp[i], xp);
    if (residual) Elt<T>::unpack(vq[i], xq);
#pragma unroll
    for (int j = 0; j < P; ++j) {
      const float w = f(xp[j], residual ? xq[j] : 0.f);
      my += static_cast<double>(w);
      if (w > 0.f) last_nz = i * P + j;
    }
  }
  double ctot;
  const double cincl = block_inclusive_scan(my, &ctot);
  const double cexcl = cincl - my;
  if (threadIdx.x == 0) s_tok = -1;
  __syncthreads();
  if (cexcl <= local && cincl > local) {
    double run = cexcl;
    int tok = -1;
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
    if (tok < 0) tok = last_nz;  // rounding inside the owning thread
    s_tok = tok;
  }
  __syncthreads();
  int tok = s_tok;
  if (tok < 0) tok = block_max_int(last_nz);  // u*Z beyond the chunk total
  if (threadIdx.x == 0) {
    if (tok < 0) tok = 0;
    p.out_tokens[b * (g + 1) + s.n] = chunk * p.CE + tok;
  }
}

}  // namespace specv
