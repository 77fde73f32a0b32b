// sparse.cuh — verification against sparse draft rows (the output of the
// centroid-masked draft head, centroid.cuh).
//
// Draft row j of sequence b is a list of candidates (token ids ascending,
// logits); q_j is the softmax of the candidates' logits / T and 0 off the
// candidates ("Gemma 4 Multi-Token Prediction (MTP) 深度解析" §3.4; the
// acceptance rule is unchanged, §2.2: accept iff u < p(d)/q(d), q(d) = 0
// accepting).  The chain is the row reducer over the target rows only (the
// draft rows are never streamed) and sparse_tail_kernel, grid (parts, B):
//   * every CTA of a sequence folds the target partials, computes the draft
//     rows' normalisers from their candidates, looks the drafts up in the
//     candidate lists (a 32-way warp search) and decides;
//   * after a rejection at n, the residual max(0, p_n - q_n) puts p_n's own
//     mass on every non-candidate token.  The mass of a vocabulary chunk is
//     sum_x p_n(x) - sum_{candidates x in the chunk} min(p_n(x), q_n(x)), both
//     in two-float arithmetic (the same rounded p_n(x) enters both sums), so
//     only the target row n is re-read;
//   * the last CTA draws: the chunk from the chunk masses, then the entry with
//     the chunk's candidates scattered into a shared-memory q map.
#pragma once

#include <cfloat>
#include <climits>

#include "common.cuh"
#include "decide.cuh"
#include "rowstats.cuh"
#include "sample.cuh"

namespace specv {

constexpr int kSparseThreads = 512;
constexpr int kSparseWarps = kSparseThreads / 32;
constexpr int kSparseStage = 2048;  // candidates of a CTA's chunk range staged in shared memory

struct SparseParams {
  const void* target;          // [B, gamma+1, V]
  const int32_t* cand_tok;     // [B*gamma, stride], ascending within a row
  const float* cand_logit;     // [B*gamma, stride]
  const int32_t* cand_count;   // [B*gamma]
  const float* u_resample;     // [B]
  const float4* partials;      // target-row partials of the row reducer
  float* mass;                 // [B, cpr] chunk masses of the row (pair) drawn from
  int32_t* cand_lo;            // [B, cpr+1] first candidate of each chunk of row n
  int* tail_done;              // [B * kCounterStride]
  DecideParams dp;             // dp.draft is unused
  int B, gamma, V, CE, cpr, stride;
};

// Loads a[i] from global memory (an input) or from shared memory.
struct GlobalI32 {
  const int32_t* a;
  __device__ __forceinline__ int operator()(int i) const { return __ldg(a + i); }
};
struct SmemI32 {
  const int32_t* a;
  __device__ __forceinline__ int operator()(int i) const { return a[i]; }
};

// Warp-wide lower bound in an ascending array of n entries: the first index
// i with a(i) >= key (n if none).  A 32-way search: each round every lane
// reads the start of one of 32 segments, so 8,192 entries take three rounds
// of reads.
template <typename A>
__device__ __forceinline__ int warp_lower_bound(const A& a, int n, int key) {
  const int lane = threadIdx.x & 31;
  int lo = 0, len = n;
  while (len > 32) {
    const int seg = (len + 31) / 32;
    const bool below = (lane * seg < len) && (a(lo + lane * seg) < key);
    const int L = __popc(__ballot_sync(0xffffffffu, below));  // segments starting below key
    if (L == 0) return lo;
    lo += (L - 1) * seg;  // the boundary lies in segment L-1 or at its end
    len = min(seg, len - (L - 1) * seg);
  }
  const bool below = (lane < len) && (a(lo + lane) < key);
  return lo + __popc(__ballot_sync(0xffffffffu, below));
}

// Two-float warp reduction (every lane gets the sum).
__device__ __forceinline__ F2 warp_sum_f2(F2 v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const F2 o{__shfl_xor_sync(0xffffffffu, v.hi, off), __shfl_xor_sync(0xffffffffu, v.lo, off)};
    v = f2_add(v, o);
  }
  return v;
}

// Statistics of a sparse draft row, warp-wide: mk = fl(max logit * ks) and
// log2 of sum 2^(fma(l, ks, -mk)) over the candidates (compensated sums).
__device__ __forceinline__ RowStat cand_row_stats(const float* lg, int n, float ks) {
  const int lane = threadIdx.x & 31;
  float m = -FLT_MAX;
  for (int i = lane; i < n; i += 32) m = fmaxf(m, __ldg(lg + i));
  m = warp_max(m);
  const float mk = m * ks;
  float s = 0.f, c = 0.f;
  for (int i = lane; i < n; i += 32) neumaier_add(s, c, ex2(fmaf(__ldg(lg + i), ks, -mk)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, s, off);
    const float oc = __shfl_xor_sync(0xffffffffu, c, off);
    neumaier_add(s, c, os);
    c += oc;
  }
  RowStat st;
  st.mk = (n > 0) ? mk : kNegHuge;
  st.argmax = -1;
  st.pad = 0;
  st.lse2 = log2f(s + c);
  return st;
}

// Normalised weights of the residual row pair: p_n(x) from a target logit,
// q_n(x) from a candidate's logit (explicitly rounded operations: every
// evaluation of the same entry gives the same bits).
struct SparseW {
  float ks, mkp, invSp, mkq, invSq;
  __device__ __forceinline__ float p(float xp) const { return __fmul_rn(ex2(fmaf(xp, ks, -mkp)), invSp); }
  __device__ __forceinline__ float q(float lq) const { return __fmul_rn(ex2(fmaf(lq, ks, -mkq)), invSq); }
};

// Candidates of draft row `row` (the caller's count, clamped to [0, stride]).
__device__ __forceinline__ int cand_n(const SparseParams& p, int row) {
  return min(max(__ldg(p.cand_count + row), 0), p.stride);
}

template <typename T>
__device__ __forceinline__ float load_logit(const void* base, size_t idx) {
  return Elt<T>::load1(base, idx);
}

// Level 2 of a sparse draw, block-wide: the entry of chunk `chunk` at which
// the running weight passes `local` (the beyond-total marker, or no crossing
// by rounding: the chunk's last entry of nonzero weight).  residual: weights
// p_n(x) - min(p_n(x), q(x)) with q from the shared-memory map (0 off the
// candidates); otherwise the plain row's 2^(fma(x, ks, -mk)).
template <typename T>
__device__ __forceinline__ int sparse_entry(const SparseParams& p, size_t rowp, int chunk, bool residual,
                                            const SparseW& f, float plain_mk, const float* qmap, F2 local) {
  constexpr int P = Elt<T>::kPerVec;
  __shared__ F2 s_wtot[kSparseWarps];
  __shared__ int s_first, s_lastnz, s_tok;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const uint4* vp = chunk_vec<T>(p.target, rowp, p.V, chunk, p.CE);
  const int nvec = min(p.CE, p.V - chunk * p.CE) / P;
  float w[P];
  F2 my = f2_from(0.f);
  int last_nz = -1;
  {
    const uint4 a = (t < nvec) ? __ldg(vp + t) : neg_inf_vec<T>();
    float xp[P];
    Elt<T>::unpack(a, xp);
#pragma unroll
    for (int k = 0; k < P; ++k) {
      float x = 0.f;
      if (t < nvec) {
        if (residual) {
          const float pp = f.p(xp[k]);
          x = __fsub_rn(pp, fminf(pp, qmap[t * P + k]));
        } else {
          x = ex2(fmaf(xp[k], f.ks, -plain_mk));
        }
      }
      w[k] = x;
      my = f2_add(my, f2_from(x));
      if (x > 0.f) last_nz = t * P + k;
    }
  }
  if (t == 0) {
    s_first = INT_MAX;
    s_lastnz = -1;
  }
  F2 incl = warp_scan_incl(my);
  if (lane == 31) s_wtot[warp] = incl;
  __syncthreads();
  F2 wt = (lane < kSparseWarps) ? s_wtot[lane] : f2_from(0.f);
  wt = warp_scan_incl(wt);
  const F2 wpre = f2_shfl(wt, warp > 0 ? warp - 1 : 0);
  if (warp > 0) incl = f2_add(incl, wpre);
  if (f2_gt(incl, local)) atomicMin(&s_first, t);
  if (last_nz >= 0) atomicMax(&s_lastnz, last_nz);
  __syncthreads();
  const int first = s_first;
  if (t == first) {
    F2 run = f2_sub(incl, my);
    int tok = -1;
#pragma unroll
    for (int k = 0; k < P; ++k) {
      run = f2_add(run, f2_from(w[k]));
      if (tok < 0 && f2_gt(run, local)) tok = t * P + k;
    }
    s_tok = (tok >= 0) ? tok : ((last_nz >= 0) ? last_nz : max(s_lastnz, 0));
  } else if (first == INT_MAX && t == 0) {
    s_tok = max(s_lastnz, 0);
  }
  __syncthreads();
  return s_tok;
}

template <typename T>
__global__ void __launch_bounds__(kSparseThreads, 1) sparse_tail_kernel(const __grid_constant__ SparseParams p) {
  __shared__ RowStat rs[2 * 31 + 1];
  __shared__ SeqState s_seq;
  __shared__ float s_xq[32];
  __shared__ int s_lo, s_hi, s_last;
  __shared__ int32_t st_tok[kSparseStage];
  __shared__ float st_q[kSparseStage];
  __shared__ float sm_mass[4096];
  __shared__ float qmap[2048];
  const int b = blockIdx.y, part = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.gamma, slots = 2 * g + 1;
  const bool greedy = seq_is_greedy(p.dp.temperature, b);
  const float ks = greedy ? 0.f : kLog2e / p.dp.temperature[b];

  // ---- inputs of the decision (none comes from the row reducer) ----
  DecideIn din;
  if (warp == 0) {
    din.d = -1;
    din.xp = din.xq = din.u = 0.f;
    if (lane < g) {
      din.d = p.dp.draft_tokens[b * g + lane];
      if (!greedy && din.d >= 0 && din.d < p.V) {
        din.xp = Elt<T>::load1(p.target, (static_cast<size_t>(b) * (g + 1) + lane) * p.V + din.d);
        din.u = p.dp.u_accept[b * g + lane];
      }
    }
  } else if (!greedy) {
    // the drafts' own logits: a search of each candidate list (-inf if absent)
    for (int j = warp - 1; j < g; j += kSparseWarps - 1) {
      const int row = b * g + j;
      const int d = p.dp.draft_tokens[row];
      const int n = cand_n(p, row);
      const int32_t* tok = p.cand_tok + static_cast<size_t>(row) * p.stride;
      const int i = warp_lower_bound(GlobalI32{tok}, n, d);
      const bool hit = (i < n) && __ldg(tok + i) == d;
      if (lane == 0) s_xq[j] = hit ? __ldg(p.cand_logit + static_cast<size_t>(row) * p.stride + i) : -INFINITY;
    }
  }
  const float u_res = greedy ? 0.f : p.u_resample[b];
  grid_dep_wait();

  // ---- target rows from the partials, draft rows from their candidates ----
  for (int r = warp; r < (greedy ? g + 1 : slots); r += kSparseWarps) {
    RowStat st;
    if (r <= g) {
      st = combine_row<4>(p.partials + static_cast<size_t>(b * slots + r) * p.cpr, p.cpr, !greedy);
    } else {
      const int row = b * g + (r - g - 1);
      st = cand_row_stats(p.cand_logit + static_cast<size_t>(row) * p.stride, cand_n(p, row), ks);
    }
    if (lane == 0) rs[r] = st;
  }
  __syncthreads();
  if (warp == 0) {
    if (lane < g && !greedy) din.xq = s_xq[lane];
    decide_sequence<T>(p.dp, b, rs, din, part == 0, &s_seq);
  }
  __syncthreads();
  if (part == 0 && p.dp.out_debug != nullptr && !greedy && threadIdx.x < g &&
      cand_n(p, b * g + threadIdx.x) == 0) {
    // a row without candidates: q = 0 everywhere, log-normaliser -inf
    float* dbg = p.dp.out_debug + (static_cast<size_t>(b) * (g + 1) + threadIdx.x) * 4;
    dbg[1] = 0.f;
    dbg[3] = -INFINITY;
  }
  const SeqState s = s_seq;
  if (s.mode != kModeResidual && s.mode != kModeBonus) return;

  const int per = (p.cpr + gridDim.x - 1) / gridDim.x;
  const int c0 = min(p.cpr, part * per), c1 = min(p.cpr, c0 + per);
  float* mass = p.mass + static_cast<size_t>(b) * p.cpr;
  int32_t* clo = p.cand_lo + static_cast<size_t>(b) * (p.cpr + 1);
  const int drow = b * g + s.n;
  const int32_t* tok = p.cand_tok + static_cast<size_t>(drow) * p.stride;
  const float* lg = p.cand_logit + static_cast<size_t>(drow) * p.stride;
  SparseW f;
  f.ks = s.ks;
  f.mkp = rs[s.n].mk;
  f.invSp = ex2(-rs[s.n].lse2);
  f.mkq = rs[g + 1 + s.n].mk;
  f.invSq = ex2(-rs[g + 1 + s.n].lse2);
  const size_t rowp_n = static_cast<size_t>(b) * (g + 1) + s.n;

  if (s.mode == kModeResidual) {
    const int ncand = cand_n(p, drow);
    // ---- this CTA's candidates, staged with their q ----
    if (warp == 0) {
      const int lo = warp_lower_bound(GlobalI32{tok}, ncand, c0 * p.CE);
      if (lane == 0) s_lo = lo;
    } else if (warp == 1) {
      const int hi = warp_lower_bound(GlobalI32{tok}, ncand, c1 * p.CE);
      if (lane == 0) s_hi = hi;
    }
    __syncthreads();
    const int lo = s_lo, nst = s_hi - s_lo;
    const bool staged = nst <= kSparseStage;
    if (staged) {
      for (int i = threadIdx.x; i < nst; i += kSparseThreads) {
        st_tok[i] = __ldg(tok + lo + i);
        st_q[i] = f.q(__ldg(lg + lo + i));
      }
    }
    __syncthreads();
    // ---- chunk masses: one warp per chunk ----
    for (int c = c0 + warp; c < c1; c += kSparseWarps) {
      int a, e;
      if (staged) {
        a = warp_lower_bound(SmemI32{st_tok}, nst, c * p.CE);
        e = warp_lower_bound(SmemI32{st_tok}, nst, (c + 1) * p.CE);
      } else {
        a = warp_lower_bound(GlobalI32{tok + lo}, nst, c * p.CE);
        e = warp_lower_bound(GlobalI32{tok + lo}, nst, (c + 1) * p.CE);
      }
      // sum of p_n over the chunk
      constexpr int P = Elt<T>::kPerVec;
      const uint4* vp = chunk_vec<T>(p.target, rowp_n, p.V, c, p.CE);
      const int nvec = min(p.CE, p.V - c * p.CE) / P;
      uint4 v[kVecPerLane];
#pragma unroll
      for (int j = 0; j < kVecPerLane; ++j) {
        const int k = lane + 32 * j;
        v[j] = (k < nvec) ? __ldg(vp + k) : neg_inf_vec<T>();
      }
      F2 sp = f2_from(0.f);
#pragma unroll
      for (int j = 0; j < kVecPerLane; ++j) {
        float xp[P];
        Elt<T>::unpack(v[j], xp);
#pragma unroll
        for (int k = 0; k < P; ++k) sp = f2_add(sp, f2_from(f.p(xp[k])));
      }
      // minus min(p_n, q_n) over the chunk's candidates
      F2 sm = f2_from(0.f);
      for (int i = a + lane; i < e; i += 32) {
        const int x = staged ? st_tok[i] : __ldg(tok + lo + i);
        if (x < 0 || x >= p.V) continue;  // not a token: no weight to take off
        const float q = staged ? st_q[i] : f.q(__ldg(lg + lo + i));
        const float pp = f.p(load_logit<T>(p.target, rowp_n * p.V + x));
        sm = f2_add(sm, f2_from(fminf(pp, q)));
      }
      sp = warp_sum_f2(sp);
      sm = warp_sum_f2(sm);
      const F2 d = f2_sub(sp, sm);
      if (lane == 0) {
        mass[c] = fmaxf(0.f, d.hi + d.lo);
        clo[c] = lo + a;
      }
    }
    if (c1 == p.cpr && threadIdx.x == 0) clo[p.cpr] = ncand;
  } else {  // bonus: masses of p_gamma from the row partials
    const float4* Pt = p.partials + static_cast<size_t>(b * slots + g) * p.cpr;
    const float mk = rs[g].mk;
    for (int c = c0 + threadIdx.x; c < c1; c += kSparseThreads) {
      const float4 q = __ldcg(Pt + c);
      mass[c] = q.y * ex2(q.w - mk);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(&p.tail_done[b * kCounterStride], 1);
    s_last = (old == static_cast<int>(gridDim.x) - 1);
    if (s_last) p.tail_done[b * kCounterStride] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- the draw (last CTA): level 1, the chunk ----
  const bool staged_m = p.cpr <= 4096;
  if (staged_m) {
    for (int c = threadIdx.x; c < p.cpr; c += kSparseThreads) sm_mass[c] = __ldcg(mass + c);
    __syncthreads();
  }
  __shared__ int s_chunk, s_resid;
  __shared__ F2 s_local;
  if (warp == 0) {
    bool residual = (s.mode == kModeResidual);
    F2 local;
    int chunk;
    MassScan ms = staged_m ? scan_masses_fn(SmemMass{sm_mass}, p.cpr) : scan_masses(mass, p.cpr);
    if (residual && !(ms.Z.hi > 0.f)) {
      // Z == 0 cannot happen in exact arithmetic: draw from p_n itself
      const PartialMass pn{p.partials + static_cast<size_t>(b * slots + s.n) * p.cpr, rs[s.n].mk};
      ms = scan_masses_fn(pn, p.cpr);
      chunk = pick_chunk_fn(pn, ms, f2_mul_f(ms.Z, u_res), &local);
      residual = false;
    } else if (staged_m) {
      chunk = pick_chunk_fn(SmemMass{sm_mass}, ms, f2_mul_f(ms.Z, u_res), &local);
    } else {
      chunk = pick_chunk(mass, ms, f2_mul_f(ms.Z, u_res), &local);
    }
    if (lane == 0) {
      s_chunk = chunk;
      s_local = local;
      s_resid = residual;
    }
  }
  __syncthreads();
  const int chunk = s_chunk;
  const bool residual = s_resid;
  // ---- level 2: the chunk's candidates scattered into the q map ----
  if (residual) {
    for (int i = threadIdx.x; i < p.CE; i += kSparseThreads) qmap[i] = 0.f;
    __syncthreads();
    const int a = __ldcg(clo + chunk), e = __ldcg(clo + chunk + 1);
    for (int i = a + threadIdx.x; i < e; i += kSparseThreads) {
      const int o = __ldg(tok + i) - chunk * p.CE;
      if (o >= 0 && o < p.CE) qmap[o] = f.q(__ldg(lg + i));
    }
    __syncthreads();
  }
  const int rowj = (s.mode == kModeResidual) ? s.n : g;  // the Z = 0 fallback keeps row n
  const int e = sparse_entry<T>(p, static_cast<size_t>(b) * (g + 1) + rowj, chunk, residual, f, rs[rowj].mk, qmap,
                                s_local);
  if (threadIdx.x == 0) p.dp.out_tokens[b * (g + 1) + s.n] = chunk * p.CE + e;
}

}  // namespace specv
