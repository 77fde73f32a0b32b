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
constexpr int kSparseRowStage = 4096;  // a row's candidate tokens staged whole (the draw's mass buffer)

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

// Partial statistics of a share [i0, i1) of a sparse draft row, warp-wide:
// the raw maximum M and s = sum 2^(fma(l, ks, -fl(M*ks))) (compensated),
// 32 entries per lane loaded at once.  Shares combine like the row
// reducer's chunk partials.
struct CandPartial {
  float M, s;
};

__device__ __forceinline__ CandPartial cand_partial(const float* lg, int i0, int i1, float ks) {
  const int lane = threadIdx.x & 31;
  constexpr int kBlk = 32;  // entries per lane per step
  float M = -FLT_MAX, mk = kNegHuge, s = 0.f, c = 0.f;
  for (int base = i0; base < i1; base += 32 * kBlk) {
    float x[kBlk];
#pragma unroll
    for (int q = 0; q < kBlk; ++q) {
      const int i = base + lane + 32 * q;
      x[q] = (i < i1) ? __ldg(lg + i) : -INFINITY;
    }
    float m = M;
#pragma unroll
    for (int q = 0; q < kBlk; ++q) m = fmaxf(m, x[q]);
    m = warp_max(m);
    const float nmk = m * ks;
    if (nmk != mk) {  // rescale what was summed so far (0 on the first step)
      const float sc = ex2(mk - nmk);
      s *= sc;
      c *= sc;
      mk = nmk;
    }
    M = m;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int q = 0; q < kBlk; q += 4) {
      a0 += ex2(fmaf(x[q], ks, -mk));
      a1 += ex2(fmaf(x[q + 1], ks, -mk));
      a2 += ex2(fmaf(x[q + 2], ks, -mk));
      a3 += ex2(fmaf(x[q + 3], ks, -mk));
    }
    neumaier_add(s, c, (a0 + a1) + (a2 + a3));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, s, off);
    const float oc = __shfl_xor_sync(0xffffffffu, c, off);
    neumaier_add(s, c, os);
    c += oc;
  }
  return CandPartial{M, s + c};
}

// Normalised weights of the residual row pair: p_n(x) from a target logit,
// q_n(x) from a candidate's logit (explicitly rounded operations: every
// evaluation of the same entry gives the same bits).
// Both in units of 2^mkp * S_p (the target row's scaled maximum and sum), so
// p costs one exp2: p(x) = 2^(fma(x, ks, -mkp)), q(x) = 2^(fma(l, ks, -mkq))
// * qs with qs = S_p / S_q.  Chunk masses in these units are proportional to
// the true ones, which is all the inverse CDF needs.
struct SparseW {
  float ks, mkp, mkq, qs;
  __device__ __forceinline__ float p(float xp) const { return ex2(fmaf(xp, ks, -mkp)); }
  __device__ __forceinline__ float q(float lq) const { return __fmul_rn(ex2(fmaf(lq, ks, -mkq)), qs); }
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
__device__ __forceinline__ int sparse_entry(const SparseParams& p, int chunk, bool residual, const SparseW& f,
                                            float plain_mk, const float* qmap, F2 local, uint4 a) {
  constexpr int P = Elt<T>::kPerVec;
  __shared__ F2 s_wtot[kSparseWarps];
  __shared__ int s_first, s_lastnz, s_tok;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int nvec = min(p.CE, p.V - chunk * p.CE) / P;
  float w[P];
  F2 my = f2_from(0.f);
  int last_nz = -1;
  {  // a: vector t of the chunk, loaded by the caller
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
  __shared__ CandPartial s_cp[31 * kSparseWarps];
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
  }
  const float u_res = greedy ? 0.f : p.u_resample[b];
  grid_dep_wait();

  // ---- target rows from the partials (warps 0..gamma); meanwhile the other
  // warps look the drafts up in their candidate lists (-inf if absent) ----
  for (int r = warp; r <= g; r += kSparseWarps) {
    const RowStat st = combine_row<4>(p.partials + static_cast<size_t>(b * slots + r) * p.cpr, p.cpr, !greedy);
    if (lane == 0) rs[r] = st;
  }
  if (!greedy) {
    const int w0 = (g + 1 < kSparseWarps) ? g + 1 : 0;  // with gamma >= 15 every warp takes a share
    for (int j = warp - w0; warp >= w0 && j < g; j += kSparseWarps - w0) {
      const int row = b * g + j;
      const int d = p.dp.draft_tokens[row];
      const int n = cand_n(p, row);
      const int32_t* tok = p.cand_tok + static_cast<size_t>(row) * p.stride;
      const int i = warp_lower_bound(GlobalI32{tok}, n, d);
      const bool hit = (i < n) && __ldg(tok + i) == d;
      if (lane == 0) s_xq[j] = hit ? __ldg(p.cand_logit + static_cast<size_t>(row) * p.stride + i) : -INFINITY;
    }
  }
  // ---- draft rows from their candidates: each row split over wpr warps ----
  if (!greedy) {
    const int wpr = max(1, kSparseWarps / g);
    for (int jj = warp / wpr; jj < g && warp < wpr * g; jj += kSparseWarps / wpr) {
      const int row = b * g + jj, k = warp % wpr;
      const int n = cand_n(p, row);
      const CandPartial cp =
          cand_partial(p.cand_logit + static_cast<size_t>(row) * p.stride, n * k / wpr, n * (k + 1) / wpr, ks);
      if (lane == 0) s_cp[jj * kSparseWarps + k] = cp;
    }
  }
  __syncthreads();
  if (!greedy && threadIdx.x < g) {
    // fold the shares of draft row jj: rescale each to the row's scaled maximum
    const int jj = threadIdx.x, wpr = max(1, kSparseWarps / g);
    float M = -FLT_MAX;
    for (int k = 0; k < wpr; ++k) M = fmaxf(M, s_cp[jj * kSparseWarps + k].M);
    const float mk = M * ks;
    float sum = 0.f, c = 0.f;
    for (int k = 0; k < wpr; ++k) {
      const CandPartial cp = s_cp[jj * kSparseWarps + k];
      if (cp.s > 0.f) neumaier_add(sum, c, cp.s * ex2(cp.M * ks - mk));
    }
    RowStat st;
    st.mk = (cand_n(p, b * g + jj) > 0) ? mk : kNegHuge;
    st.argmax = -1;
    st.pad = 0;
    st.lse2 = log2f(sum + c);
    rs[g + 1 + jj] = st;
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
  f.mkq = rs[g + 1 + s.n].mk;
  f.qs = ex2(rs[s.n].lse2 - rs[g + 1 + s.n].lse2);
  const size_t rowp_n = static_cast<size_t>(b) * (g + 1) + s.n;

  if (s.mode == kModeResidual) {
    const int ncand = cand_n(p, drow);
    // ---- the candidates: the whole row's tokens in shared memory when they
    // fit (the draw's mass buffer, free until then: one load round, and every
    // search after it is in shared memory; the q values are loaded with the
    // chunk's logits); otherwise this CTA's share, found by searches in
    // global memory and staged with its q ----
    int32_t* rowtok = reinterpret_cast<int32_t*>(sm_mass);
    const bool whole = ncand <= kSparseRowStage;
    int lo = 0, nst = ncand;
    bool staged = true;
    if (whole) {
      constexpr int kPer = kSparseRowStage / kSparseThreads;
      int32_t tv[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = static_cast<int>(threadIdx.x) + j * kSparseThreads;
        tv[j] = (i < ncand) ? __ldg(tok + i) : 0;
      }
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = static_cast<int>(threadIdx.x) + j * kSparseThreads;
        if (i < ncand) rowtok[i] = tv[j];
      }
    } else {
      if (warp == 0) {
        const int l = warp_lower_bound(GlobalI32{tok}, ncand, c0 * p.CE);
        if (lane == 0) s_lo = l;
      } else if (warp == 1) {
        const int h = warp_lower_bound(GlobalI32{tok}, ncand, c1 * p.CE);
        if (lane == 0) s_hi = h;
      }
      __syncthreads();
      lo = s_lo;
      nst = s_hi - s_lo;
      staged = nst <= kSparseStage;
      if (staged) {
        for (int i = threadIdx.x; i < nst; i += kSparseThreads) {
          st_tok[i] = __ldg(tok + lo + i);
          st_q[i] = f.q(__ldg(lg + lo + i));
        }
      }
    }
    __syncthreads();
    const int32_t* stok = whole ? rowtok : st_tok;  // staged tokens, from index lo
    // ---- chunk masses: one warp per chunk ----
    for (int c = c0 + warp; c < c1; c += kSparseWarps) {
      int a, e;
      if (staged) {
        a = warp_lower_bound(SmemI32{stok}, nst, c * p.CE);
        e = warp_lower_bound(SmemI32{stok}, nst, (c + 1) * p.CE);
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
      // this lane's first candidate of the chunk, gathered with the vectors
      // (a chunk holds about 32 candidates: usually the only one)
      int x0 = -1;
      float xp0 = 0.f, q0 = 0.f;
      if (a + lane < e) {
        x0 = staged ? stok[a + lane] : __ldg(tok + lo + a + lane);
        q0 = (staged && !whole) ? st_q[a + lane] : f.q(__ldg(lg + lo + a + lane));
        if (x0 >= 0 && x0 < p.V) xp0 = load_logit<T>(p.target, rowp_n * p.V + x0);
      }
      // compensated (Neumaier) sums per lane, four independent chains;
      // lanes combine in two-float
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, ca[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < kVecPerLane; ++j) {
        float xp[P];
        Elt<T>::unpack(v[j], xp);
#pragma unroll
        for (int k = 0; k < P; ++k) neumaier_add(sa[k & 3], ca[k & 3], f.p(xp[k]));
      }
      F2 sp = f2_from(0.f);
#pragma unroll
      for (int k = 0; k < 4; ++k) sp = f2_add(sp, f2_add(f2_from(sa[k]), f2_from(ca[k])));
      // minus min(p_n, q_n) over the chunk's candidates
      float s1 = 0.f, c1m = 0.f;
      if (x0 >= 0 && x0 < p.V) neumaier_add(s1, c1m, fminf(f.p(xp0), q0));
      for (int i = a + lane + 32; i < e; i += 32) {
        const int x = staged ? stok[i] : __ldg(tok + lo + i);
        if (x < 0 || x >= p.V) continue;  // not a token: no weight to take off
        const float q = (staged && !whole) ? st_q[i] : f.q(__ldg(lg + lo + i));
        const float pp = f.p(load_logit<T>(p.target, rowp_n * p.V + x));
        neumaier_add(s1, c1m, fminf(pp, q));
      }
      F2 sm = f2_add(f2_from(s1), f2_from(c1m));
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
  if (threadIdx.x == 0) s_last = last_cta_arrives(&p.tail_done[b * kCounterStride], gridDim.x);
  __syncthreads();
  if (!s_last) return;

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
  const int rowj = (s.mode == kModeResidual) ? s.n : g;  // the Z = 0 fallback keeps row n
  uint4 av;  // vector t of the chosen chunk: loaded now, used after the map is built
  {
    constexpr int P = Elt<T>::kPerVec;
    const uint4* vp = chunk_vec<T>(p.target, static_cast<size_t>(b) * (g + 1) + rowj, p.V, chunk, p.CE);
    const int nvec = min(p.CE, p.V - chunk * p.CE) / P;
    av = (static_cast<int>(threadIdx.x) < nvec) ? __ldg(vp + threadIdx.x) : neg_inf_vec<T>();
  }
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
  const int e = sparse_entry<T>(p, chunk, residual, f, rs[rowj].mk, qmap, s_local, av);
  if (threadIdx.x == 0) p.dp.out_tokens[b * (g + 1) + s.n] = chunk * p.CE + e;
}

}  // namespace specv
