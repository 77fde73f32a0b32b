// sample.cuh — the tail kernel: decide, residual normaliser, inverse-CDF draw.
//
// tail_kernel, grid (parts, B), one sequence per blockIdx.y.  Every CTA of a
// sequence folds the sequence's row partials (a few KB from L2) and takes the
// acceptance decision (decide.cuh) — identical in every CTA, so no CTA waits
// on another; part 0 writes the outputs.  Then, when the sequence samples:
//   * after a rejection at position n the token is drawn from
//     w(x) = max(0, p_n(x) - q_n(x)) / Z ("Gemma 4 Multi-Token Prediction
//     (MTP) 深度解析" §2.2; "自投机解码：层跳过与拒绝采样实现大模型推理加速" §3.2):
//     each CTA computes the masses of w over its share of the chunks, one warp
//     per chunk over the row pair;
//   * after a fully accepted draft the bonus is drawn from p_gamma ("第 8 章
//     投机解码：一次前向，验证好几个字", 多出来的那一个 token 从哪来): the chunk masses
//     come straight from the row partials.
// The last CTA of the sequence to finish (a per-sequence counter, reset by
// that CTA) draws the token by inverse CDF in ascending vocabulary order, the
// smallest k with sum_{x<=k} w(x) > u*Z: one warp scans the chunk masses to
// pick the chunk, then scans that chunk's entries.  Element weights are fp32;
// running sums across lanes and chunks are two-float (F2) sums, since FP64 is
// slow on GB300.
#pragma once

#include <cfloat>
#include <climits>

#include "common.cuh"
#include "decide.cuh"
#include "rowstats.cuh"

namespace specv {

constexpr int kTailThreads = 512;
constexpr int kTailWarps = kTailThreads / 32;

struct SampleParams {
  const void* target;
  const void* draft;
  const float* u_resample;
  const float4* partials;  // [B*(2*gamma+1)*cpr] from the row reducer
  float* mass;             // [B*cpr] chunk masses of the selected row (pair)
  int* tail_done;          // [B*kCounterStride] CTAs finished per sequence
  DecideParams dp;
  int B, gamma, V, CE, cpr;
};

// Weight of one vocabulary entry of the selected row (pair), in the units of
// the chunk masses: residual -> max(0, p - q); plain row -> p * S (units of
// 2^mk).
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

__device__ __forceinline__ WeightFn make_weight(const RowStat& rp, const RowStat& rq, bool residual,
                                                float ks) {
  WeightFn f;
  f.ks = ks;
  f.residual = residual;
  f.mkp = rp.mk;
  f.invSp = ex2(-rp.lse2);
  f.mkq = residual ? rq.mk : 0.f;
  f.invSq = residual ? ex2(-rq.lse2) : 0.f;
  return f;
}

template <typename T>
__device__ __forceinline__ const uint4* chunk_vec(const void* base, size_t row, int V, int c, int CE) {
  return reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(base) +
                                        (row * V + static_cast<size_t>(c) * CE) * sizeof(T));
}

// Two-float numbers (hi + lo, |lo| <= ulp(hi)/2): sums to about 2^-44
// relative in fp32 arithmetic, since FP64 is slow on GB300.
struct F2 {
  float hi, lo;
};
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b.hi - bb);  // exact error of s
  const float t = e + a.lo + b.lo;
  const float h = s + t;
  return F2{h, t - (h - s)};
}
__device__ __forceinline__ F2 f2_from(float x) { return F2{x, 0.f}; }
__device__ __forceinline__ F2 f2_mul_f(F2 a, float u) {  // a * u
  const float h = a.hi * u;
  const float l = fmaf(a.hi, u, -h) + a.lo * u;
  const float r = h + l;
  return F2{r, l - (r - h)};
}
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) { return f2_add(a, F2{-b.hi, -b.lo}); }
__device__ __forceinline__ bool f2_gt(F2 a, F2 b) { return (a.hi - b.hi) + (a.lo - b.lo) > 0.f; }
__device__ __forceinline__ F2 f2_shfl_up(F2 v, int off) {
  return F2{__shfl_up_sync(0xffffffffu, v.hi, off), __shfl_up_sync(0xffffffffu, v.lo, off)};
}
__device__ __forceinline__ F2 f2_shfl(F2 v, int src) {
  return F2{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}
// Warp-inclusive scan of one two-float per lane.
__device__ __forceinline__ F2 warp_scan_incl(F2 v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const F2 o = f2_shfl_up(v, off);
    if (lane >= off) v = f2_add(v, o);
  }
  return v;
}

// Mass of w over one chunk (warp-wide; lanes hold vectors lane, lane+32, ...).
template <typename T>
__device__ __forceinline__ float chunk_mass(const SampleParams& p, const WeightFn& f, int b, int n,
                                            int c) {
  constexpr int P = Elt<T>::kPerVec;
  const int lane = threadIdx.x & 31, g = p.gamma;
  const uint4* vp = chunk_vec<T>(p.target, static_cast<size_t>(b) * (g + 1) + n, p.V, c, p.CE);
  const uint4* vq = chunk_vec<T>(p.draft, static_cast<size_t>(b) * g + n, p.V, c, p.CE);
  const int nvec = min(p.CE, p.V - c * p.CE) / P;
  uint4 a[kVecPerLane], q[kVecPerLane];
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    const int k = lane + 32 * j;
    a[j] = (k < nvec) ? __ldg(vp + k) : neg_inf_vec<T>();
    q[j] = (k < nvec) ? __ldg(vq + k) : neg_inf_vec<T>();
  }
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    float xp[P], xq[P];
    Elt<T>::unpack(a[j], xp);
    Elt<T>::unpack(q[j], xq);
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < P; ++k) t += f(xp[k], xq[k]);
    acc += t;
  }
  return warp_sum(acc);
}

// Level 1 of the inverse-CDF draw, warp-wide.  Lane l owns the contiguous
// chunk range [c0, c1) of the chunk masses mass(c); the scan gives each lane
// its own sum and the inclusive sum over lanes, and Z the total.
struct MassScan {
  F2 lsum, incl, Z;
  int c0, c1;
};
template <typename MassFn>
__device__ __forceinline__ MassScan scan_masses_fn(const MassFn& mass, int n) {
  const int lane = threadIdx.x & 31;
  const int per = (n + 31) / 32;
  MassScan ms;
  ms.c0 = min(n, lane * per);
  ms.c1 = min(n, ms.c0 + per);
  ms.lsum = f2_from(0.f);
#pragma unroll 4
  for (int c = ms.c0; c < ms.c1; ++c) ms.lsum = f2_add(ms.lsum, f2_from(mass(c)));
  ms.incl = warp_scan_incl(ms.lsum);
  ms.Z = f2_shfl(ms.incl, 31);
  return ms;
}

// The chunk holding `target` (= u*Z): the smallest c whose inclusive prefix
// exceeds it.  *local receives target minus the mass before that chunk, or
// FLT_MAX when rounding puts the target at or beyond the total, in which case
// the last chunk of nonzero mass is taken.
template <typename MassFn>
__device__ __forceinline__ int pick_chunk_fn(const MassFn& mass, const MassScan& ms, F2 target, F2* local) {
  const int lane = threadIdx.x & 31;
  const unsigned over = __ballot_sync(0xffffffffu, f2_gt(ms.incl, target));
  int chunk = -1;
  F2 loc = F2{FLT_MAX, 0.f};
  if (over) {
    const int L = __ffs(over) - 1;
    if (lane == L) {
      F2 run = f2_sub(ms.incl, ms.lsum);
      for (int c = ms.c0; c < ms.c1; ++c) {
        const F2 nxt = f2_add(run, f2_from(mass(c)));
        if (f2_gt(nxt, target)) {
          chunk = c;
          loc = f2_sub(target, run);
          break;
        }
        run = nxt;
      }
      if (chunk < 0) {  // rounding inside the lane: its last nonzero chunk
        for (int c = ms.c1 - 1; c >= ms.c0; --c)
          if (mass(c) > 0.f) {
            chunk = c;
            break;
          }
      }
    }
    chunk = __shfl_sync(0xffffffffu, chunk, L);
    loc = f2_shfl(loc, L);
  }
  if (chunk < 0) {  // u*Z at or beyond the total: the last nonzero chunk
    int last = -1;
    for (int c = ms.c0; c < ms.c1; ++c)
      if (mass(c) > 0.f) last = c;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
    chunk = last < 0 ? 0 : last;
    loc = F2{FLT_MAX, 0.f};
  }
  *local = loc;
  return chunk;
}

// The same over masses held in global memory (written by other CTAs: read
// through L2).
struct GlobalMass {
  const float* m;
  __device__ __forceinline__ float operator()(int c) const { return __ldcg(m + c); }
};
__device__ __forceinline__ MassScan scan_masses(const float* mass, int n) {
  return scan_masses_fn(GlobalMass{mass}, n);
}
__device__ __forceinline__ int pick_chunk(const float* mass, const MassScan& ms, F2 target, F2* local) {
  return pick_chunk_fn(GlobalMass{mass}, ms, target, local);
}

// Chunk masses of a plain row straight from its partials {M, s, argmax, mk},
// in units of 2^mk (mk: the row's combined scaled max).
struct PartialMass {
  const float4* P;
  float mk;
  __device__ __forceinline__ float operator()(int c) const {
    const float4 q = __ldcg(P + c);
    return q.y * ex2(q.w - mk);
  }
};

// Chunk masses of a plain row from its partials {M, s, argmax, mk}, in units
// of 2^mk (mk: the row's combined scaled max); this lane's range [c0, c1).
__device__ __forceinline__ void masses_from_partials(const float4* P, float mk, float* mass, int n) {
  const int lane = threadIdx.x & 31;
  const int per = (n + 31) / 32;
  const int c0 = min(n, lane * per), c1 = min(n, c0 + per);
  for (int c = c0; c < c1; ++c) {
    const float4 q = __ldcg(P + c);
    mass[c] = q.y * ex2(q.w - mk);
  }
}

constexpr int kTailSmemChunks = 4096;  // chunk masses staged in shared memory for the draw

// Chunk masses staged in shared memory.
struct SmemMass {
  const float* m;
  __device__ __forceinline__ float operator()(int c) const { return m[c]; }
};

// The inverse-CDF draw for sequence b, by the whole (last) CTA.
// rs: the sequence's combined rows; s: its decision.
// Level 1: the CTA stages the chunk masses in shared memory and one warp
// scans them for the chunk.  Level 2: thread t takes vector t of that chunk
// (8 bf16 or 4 fp32 entries) and its weights' two-float sum; a block scan of
// those sums finds the first thread whose prefix passes u*Z minus the mass of
// the earlier chunks, and that thread walks its own entries.
template <typename T>
__device__ __forceinline__ void draw_token(const SampleParams& p, int b, const SeqState s, const RowStat* rs, float u) {
  constexpr int P = Elt<T>::kPerVec;
  __shared__ float sm_mass[kTailSmemChunks];
  __shared__ F2 s_wtot[kTailWarps];
  __shared__ F2 s_local;
  __shared__ int s_chunk, s_resid, s_first, s_lastnz;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.gamma, slots = 2 * g + 1;
  float* mass = p.mass + static_cast<size_t>(b) * p.cpr;
  const bool staged = p.cpr <= kTailSmemChunks;

  // ---- level 1: which chunk ----
  if (staged) {
    for (int c = threadIdx.x; c < p.cpr; c += kTailThreads) sm_mass[c] = __ldcg(mass + c);
    __syncthreads();
  }
  if (warp == 0) {
    bool residual = (s.mode == kModeResidual);
    F2 local;
    int chunk;
    if (staged) {
      const SmemMass sm{sm_mass};
      MassScan ms = scan_masses_fn(sm, p.cpr);
      if (residual && !(ms.Z.hi > 0.f)) {
        // Z == 0 cannot happen in exact arithmetic; if rounding produces it,
        // draw from p_n itself (chunk masses from the row partials)
        const PartialMass pn{p.partials + static_cast<size_t>(b * slots + s.n) * p.cpr, rs[s.n].mk};
        for (int c = lane; c < p.cpr; c += 32) sm_mass[c] = pn(c);
        __syncwarp();
        ms = scan_masses_fn(sm, p.cpr);
        residual = false;  // weights of target row n as a plain row
      }
      chunk = pick_chunk_fn(sm, ms, f2_mul_f(ms.Z, u), &local);
    } else {
      MassScan ms = scan_masses(mass, p.cpr);
      if (residual && !(ms.Z.hi > 0.f)) {
        masses_from_partials(p.partials + static_cast<size_t>(b * slots + s.n) * p.cpr, rs[s.n].mk, mass, p.cpr);
        ms = scan_masses(mass, p.cpr);
        residual = false;
      }
      chunk = pick_chunk(mass, ms, f2_mul_f(ms.Z, u), &local);
    }
    if (lane == 0) {
      s_chunk = chunk;
      s_local = local;
      s_resid = residual;
      s_first = INT_MAX;
      s_lastnz = -1;
    }
  }
  __syncthreads();

  // ---- level 2: which entry inside the chunk (block-wide) ----
  const int chunk = s_chunk;
  if (!in_bounds(chunk >= 0 && chunk < p.cpr, p.dp.status)) return;
  const bool residual = s_resid;
  const F2 local = s_local;
  const int rowp = (s.mode == kModeResidual) ? s.n : g;  // the Z = 0 fallback keeps row n
  const WeightFn f = make_weight(rs[rowp], rs[g + 1 + (residual ? s.n : 0)], residual, s.ks);
  const uint4* vp = chunk_vec<T>(p.target, static_cast<size_t>(b) * (g + 1) + rowp, p.V, chunk, p.CE);
  const uint4* vq = residual ? chunk_vec<T>(p.draft, static_cast<size_t>(b) * g + s.n, p.V, chunk, p.CE) : vp;
  const int nvec = min(p.CE, p.V - chunk * p.CE) / P;  // <= 256 vectors of 16 B
  const int t = threadIdx.x;
  float w[P];
  F2 my = f2_from(0.f);
  int last_nz = -1;
  {
    uint4 a = neg_inf_vec<T>(), q = neg_inf_vec<T>();
    if (t < nvec) {
      a = __ldg(vp + t);
      if (residual) q = __ldg(vq + t);
    }
    float xp[P], xq[P];
    Elt<T>::unpack(a, xp);
    Elt<T>::unpack(q, xq);
#pragma unroll
    for (int k = 0; k < P; ++k) {
      w[k] = (t < nvec) ? f(xp[k], xq[k]) : 0.f;
      my = f2_add(my, f2_from(w[k]));
      if (w[k] > 0.f) last_nz = t * P + k;
    }
  }
  F2 incl = warp_scan_incl(my);
  if (lane == 31) s_wtot[warp] = incl;
  __syncthreads();
  // prefix of the earlier warps' totals: every warp scans the kTailWarps
  // totals (one per lane) at once instead of adding them one by one
  F2 wt = (lane < kTailWarps) ? s_wtot[lane] : f2_from(0.f);
  wt = warp_scan_incl(wt);
  const F2 wpre = f2_shfl(wt, warp > 0 ? warp - 1 : 0);
  if (warp > 0) incl = f2_add(incl, wpre);
  // the prefix sums are non-decreasing in t: the first thread whose inclusive
  // prefix passes `local` holds the entry
  if (f2_gt(incl, local)) atomicMin(&s_first, t);
  if (last_nz >= 0) atomicMax(&s_lastnz, last_nz);
  __syncthreads();
  const int first = s_first;
  const int out_pos = b * (g + 1) + s.n;
  if (t == first) {
    F2 run = f2_sub(incl, my);
    int tok = -1;
#pragma unroll
    for (int k = 0; k < P; ++k) {
      run = f2_add(run, f2_from(w[k]));
      if (tok < 0 && f2_gt(run, local)) tok = t * P + k;
    }
    if (tok < 0) tok = (last_nz >= 0) ? last_nz : max(s_lastnz, 0);  // rounding inside the thread
    p.dp.out_tokens[out_pos] = chunk * p.CE + tok;
  } else if (first == INT_MAX && t == 0) {
    // beyond the chunk total (rounding): the chunk's last nonzero entry
    p.dp.out_tokens[out_pos] = chunk * p.CE + max(s_lastnz, 0);
  }
}

template <typename T>
__global__ void __launch_bounds__(kTailThreads, 2) tail_kernel(const __grid_constant__ SampleParams p) {
  __shared__ RowStat rs[2 * 31 + 1];  // gamma <= 31
  __shared__ SeqState s_seq;
  __shared__ int s_last;
  const int b = blockIdx.y, part = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.gamma, slots = 2 * g + 1;
  const bool greedy = (p.dp.temperature == nullptr) || seq_is_greedy(p.dp.temperature, b);
  const int nrows = greedy ? g + 1 : slots;
  // inputs of the decision do not depend on the row reducer: load them first
  DecideIn din;
  if (warp == 0) din = prefetch_decide<T>(p.dp, b, greedy);
  const float u_res = greedy ? 0.f : p.u_resample[b];  // an input: loaded before the wait too
  grid_dep_wait();

  // ---- combine the sequence's rows, one warp per row ----
  for (int r = warp; r < nrows; r += kTailWarps) {
    const RowStat st = combine_row<4>(p.partials + static_cast<size_t>(b * slots + r) * p.cpr, p.cpr, !greedy);
    if (lane == 0) rs[r] = st;
  }
  __syncthreads();
  if (warp == 0) decide_sequence<T>(p.dp, b, rs, din, part == 0, &s_seq);
  __syncthreads();
  const SeqState s = s_seq;
  if (s.mode != kModeResidual && s.mode != kModeBonus) return;
  if (!in_bounds(s.n >= 0 && s.n <= g, p.dp.status)) return;

  // ---- chunk masses of the row (pair) to draw from, this CTA's share ----
  const int per = (p.cpr + gridDim.x - 1) / gridDim.x;
  const int c0 = min(p.cpr, part * per), c1 = min(p.cpr, c0 + per);
  float* mass = p.mass + static_cast<size_t>(b) * p.cpr;
  if (s.mode == kModeResidual) {
    const WeightFn f = make_weight(rs[s.n], rs[g + 1 + s.n], true, s.ks);
    for (int c = c0 + warp; c < c1; c += kTailWarps) {
      const float m = chunk_mass<T>(p, f, b, s.n, c);
      if (lane == 0) mass[c] = m;
    }
  } else {  // bonus: masses of p_gamma from the row partials
    const float4* P = p.partials + static_cast<size_t>(b * slots + g) * p.cpr;
    const float mk = rs[g].mk;
    for (int c = c0 + threadIdx.x; c < c1; c += kTailThreads) {
      const float4 q = __ldcg(P + c);
      mass[c] = q.y * ex2(q.w - mk);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) s_last = last_cta_arrives(&p.tail_done[b * kCounterStride], gridDim.x);
  __syncthreads();
  if (!s_last) return;
  draw_token<T>(p, b, s, rs, u_res);
}

}  // namespace specv
