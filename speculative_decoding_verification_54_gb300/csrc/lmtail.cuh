// lmtail.cuh — decision and inverse-CDF draw when the target logits come
// from the fused lm_head (lmhead.cuh).
//
//   lm_decide_kernel  one CTA per sequence: combines the target rows' tile
//                     partials (lm_head epilogue) and the draft rows' chunk
//                     partials (row reducer) and decides (decide.cuh); p_j(d)
//                     uses the target logit at the draft token, read from the
//                     fp32 logits the epilogue stored for rows j < gamma.
//   lm_tail_kernel    grid (parts, B): the residual masses
//                     max(0, p_n - q_n) per 128-entry tile of the rejected
//                     position n (stored target logits against the bf16
//                     draft logits), or, after a fully accepted draft, the
//                     bonus row's tile masses from its partials; the last CTA
//                     of a sequence draws the token by inverse CDF in
//                     ascending vocabulary order: the tile from the masses,
//                     then the entry inside it.  The bonus row gamma is not
//                     stored: every CTA of a bonus sequence picks the tile
//                     from the row's tile partials and recomputes its share of
//                     the tile's 128 logits as fp32 dot products of the hidden
//                     state with W, for the last CTA to draw from.
#pragma once

#include <cfloat>
#include <cuda_bf16.h>

#include "common.cuh"
#include "decide.cuh"
#include "lmhead.cuh"
#include "sample.cuh"

namespace specv {

constexpr int kLmTailThreads = 256;
constexpr int kLmTailWarps = kLmTailThreads / 32;
constexpr int kLmMassGroup = 8;  // tiles a warp reduces at once (8 x 512 B of fp32 logits)
constexpr int kLmSmemTiles = 8192;  // tile masses staged in shared memory for the draw (V <= 1,048,576)


struct LmTailParams {
  const __nv_bfloat16* hidden;  // [R, H], R = B*(gamma+1)
  const __nv_bfloat16* W;       // [V, H]
  const __nv_bfloat16* draft;   // [B, gamma, V]
  const float* logits;          // [B, gamma, V] stored target logits (sampling sequences)
  const float4* tpart;          // target rows [R][n_tiles]
  const float4* dpart;          // row slots [B*(2*gamma+1)][cpr_d], draft slots filled
  RowStat* rowstat;             // [B*(2*gamma+1)]
  SeqState* seq;                // [B]
  float* mass;                  // [B][n_tiles]
  float* xsg;                   // [B][128] the bonus row's recomputed tile
  int* tail_done;               // [B*kCounterStride]
  const float* u_resample;
  DecideParams dp;
  int B, gamma, V, H, n_tiles, cpr_d;
};

__global__ void __launch_bounds__(kLmTailThreads) lm_decide_kernel(const __grid_constant__ LmTailParams p) {
  __shared__ RowStat rs[2 * 31 + 1];
  __shared__ SeqState s_seq;
  grid_dep_launch();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.gamma, slots = 2 * g + 1;
  const bool greedy = seq_is_greedy(p.dp.temperature, b);
  const int nrows = greedy ? g + 1 : slots;
  // inputs that the previous kernels do not write: load before waiting
  DecideIn in;
  in.d = -1;
  in.xp = in.xq = in.u = 0.f;
  bool gather = false;
  if (warp == 0 && lane < g) {
    in.d = p.dp.draft_tokens[b * g + lane];
    gather = !greedy && in.d >= 0 && in.d < p.V;
    if (gather) {
      in.xq = __bfloat162float(p.draft[(static_cast<size_t>(b) * g + lane) * p.V + in.d]);
      in.u = p.dp.u_accept[b * g + lane];
    }
  }
  grid_dep_wait();
  if (gather) in.xp = __ldcg(p.logits + (static_cast<size_t>(b) * g + lane) * p.V + in.d);
  for (int r = warp; r < nrows; r += kLmTailWarps) {
    RowStat st;
    if (r <= g)  // one partial per 128-entry tile: 2048 for a 262,144-entry row
      st = combine_row<32>(p.tpart + static_cast<size_t>(b * (g + 1) + r) * p.n_tiles, p.n_tiles, !greedy);
    else
      st = combine_row(p.dpart + static_cast<size_t>(b * slots + r) * p.cpr_d, p.cpr_d, true);
    if (lane == 0) {
      rs[r] = st;
      p.rowstat[b * slots + r] = st;
    }
  }
  __syncthreads();
  if (warp == 0) {
    decide_sequence<__nv_bfloat16>(p.dp, b, rs, in, true, &s_seq);
    if (lane == 0) p.seq[b] = s_seq;
  }
}

// Four consecutive bf16 draft logits (8-byte aligned: V % 8 == 0).
__device__ __forceinline__ void load_bf16x4(const __nv_bfloat16* src, float (&x)[4]) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
  bf16x2_unpack(u.x, x[0], x[1]);
  bf16x2_unpack(u.y, x[2], x[3]);
}

// logit = <h, W[x]> in fp32 (warp-wide; lane 0's value is the result).
__device__ __forceinline__ float dot_row(const uint4* h4, const uint4* w4, int nvec) {
  const int lane = threadIdx.x & 31;
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
  for (int i = lane; i < nvec; i += 32) {
    const uint4 a = __ldg(h4 + i), w = __ldg(w4 + i);
    float ha[8], wa[8];
    Elt<__nv_bfloat16>::unpack(a, ha);
    Elt<__nv_bfloat16>::unpack(w, wa);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      acc0 = fmaf(ha[k], wa[k], acc0);
      acc1 = fmaf(ha[k + 1], wa[k + 1], acc1);
    }
  }
  return warp_sum(acc0 + acc1);
}

// Level 1 of the inverse-CDF draw over tile masses staged in shared memory,
// by the whole CTA (every thread calls; a warp alone walked 2,048 masses 64
// per lane, about 6 K cycles): thread t owns the contiguous tiles
// [t*per, (t+1)*per), and a block scan of the two-float range sums gives each
// thread its inclusive prefix and every thread the total Z.
struct BlockMassScan {
  F2 lsum, incl, Z;
  int c0, c1;
};
__device__ __forceinline__ BlockMassScan block_scan_masses(const float* sm, int n, F2* s_w) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int per = (n + kLmTailThreads - 1) / kLmTailThreads;
  BlockMassScan bs;
  bs.c0 = min(n, t * per);
  bs.c1 = min(n, bs.c0 + per);
  bs.lsum = f2_from(0.f);
  for (int c = bs.c0; c < bs.c1; ++c) bs.lsum = f2_add(bs.lsum, f2_from(sm[c]));
  const F2 wincl = warp_scan_incl(bs.lsum);
  if (lane == 31) s_w[warp] = wincl;
  __syncthreads();
  F2 before = f2_from(0.f), Z = f2_from(0.f);
  for (int w = 0; w < kLmTailWarps; ++w) {
    const F2 x = s_w[w];
    if (w < warp) before = f2_add(before, x);
    Z = f2_add(Z, x);
  }
  __syncthreads();  // s_w free again
  bs.incl = f2_add(before, wincl);
  bs.Z = Z;
  return bs;
}

// The tile holding `target` (= u*Z), as pick_chunk_fn, by the whole CTA: the
// first thread whose inclusive prefix exceeds the target walks its tiles.
// *local: target minus the mass before that tile, or FLT_MAX when rounding
// puts the target at or beyond the total (then the last tile of nonzero mass).
__device__ __forceinline__ int block_pick_tile(const float* sm, const BlockMassScan& bs, F2 target, F2* local,
                                               int* s_i, F2* s_loc) {
  const int t = threadIdx.x;
  if (t == 0) {
    s_i[0] = INT_MAX;
    s_i[1] = -1;
  }
  __syncthreads();
  if (f2_gt(bs.incl, target)) atomicMin(&s_i[0], t);
  __syncthreads();
  const int L = s_i[0];
  if (t == L) {
    int tile = -1;
    F2 loc = F2{FLT_MAX, 0.f};
    F2 run = f2_sub(bs.incl, bs.lsum);
    for (int c = bs.c0; c < bs.c1; ++c) {
      const F2 nxt = f2_add(run, f2_from(sm[c]));
      if (f2_gt(nxt, target)) {
        tile = c;
        loc = f2_sub(target, run);
        break;
      }
      run = nxt;
    }
    if (tile < 0)  // rounding inside the range: its last nonzero tile
      for (int c = bs.c1 - 1; c >= bs.c0; --c)
        if (sm[c] > 0.f) {
          tile = c;
          break;
        }
    s_i[1] = tile;
    *s_loc = loc;
  }
  if (L == INT_MAX) {  // u*Z at or beyond the total: the last nonzero tile
    int last = -1;
    for (int c = bs.c0; c < bs.c1; ++c)
      if (sm[c] > 0.f) last = c;
    if (last >= 0) atomicMax(&s_i[1], last);
    if (t == 0) *s_loc = F2{FLT_MAX, 0.f};
  }
  __syncthreads();
  const int tile = s_i[1];
  *local = *s_loc;
  __syncthreads();  // s_i, s_loc free again
  return tile < 0 ? 0 : tile;
}

__global__ void __launch_bounds__(kLmTailThreads) lm_tail_kernel(const __grid_constant__ LmTailParams p) {
  __shared__ float xs[kLmTileV];
  __shared__ float sm_mass[kLmSmemTiles];
  __shared__ int s_last, s_chunk, s_plain;
  __shared__ F2 s_local;
  __shared__ F2 s_w[kLmTailWarps];
  __shared__ int s_pi[2];
  __shared__ F2 s_ploc;
  const int b = blockIdx.y, part = blockIdx.x;
  const bool staged = p.n_tiles <= kLmSmemTiles;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.gamma, slots = 2 * g + 1;
  grid_dep_wait();
  const SeqState s = p.seq[b];
  if (s.mode != kModeResidual && s.mode != kModeBonus) return;
  const bool residual = (s.mode == kModeResidual);
  const RowStat rp = p.rowstat[b * slots + (residual ? s.n : g)];
  const RowStat rq = residual ? p.rowstat[b * slots + g + 1 + s.n] : RowStat{};
  const WeightFn f = make_weight(rp, rq, residual, s.ks);
  float* mass = p.mass + static_cast<size_t>(b) * p.n_tiles;

  if (residual) {
    // ---- this CTA's share of the tile masses of max(0, p_n - q_n) ----
    const int per = (p.n_tiles + gridDim.x - 1) / gridDim.x;
    const int c0 = min(p.n_tiles, part * per), c1 = min(p.n_tiles, c0 + per);
    const float* lp = p.logits + (static_cast<size_t>(b) * g + s.n) * p.V;
    const __nv_bfloat16* lq = p.draft + (static_cast<size_t>(b) * g + s.n) * p.V;
    for (int t0 = c0 + warp * kLmMassGroup; t0 < c1; t0 += kLmTailWarps * kLmMassGroup) {
      float4 xp4[kLmMassGroup];
      uint2 xq2[kLmMassGroup];
#pragma unroll
      for (int j = 0; j < kLmMassGroup; ++j) {  // lane l: entries 4l..4l+3 of tile t0+j
        const int t = t0 + j;
        const size_t e = static_cast<size_t>(t) * kLmTileV + 4 * lane;
        const bool ok = t < c1 && e < static_cast<size_t>(p.V);
        xp4[j] = ok ? __ldcg(reinterpret_cast<const float4*>(lp + e))
                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        xq2[j] = ok ? __ldg(reinterpret_cast<const uint2*>(lq + e)) : make_uint2(0xff80ff80u, 0xff80ff80u);
      }
#pragma unroll
      for (int j = 0; j < kLmMassGroup; ++j) {
        float xq[4];
        bf16x2_unpack(xq2[j].x, xq[0], xq[1]);
        bf16x2_unpack(xq2[j].y, xq[2], xq[3]);
        const float w = (f(xp4[j].x, xq[0]) + f(xp4[j].y, xq[1])) + (f(xp4[j].z, xq[2]) + f(xp4[j].w, xq[3]));
        const float m = warp_sum(w);
        if (lane == 0 && t0 + j < c1) mass[t0 + j] = m;
      }
    }
  } else {
    // ---- bonus: every CTA picks the tile itself from row gamma's tile
    // partials (level 1), then recomputes its share of that tile's 128
    // logits as fp32 dot products of the hidden state with W ----
    const PartialMass pm{p.tpart + static_cast<size_t>(b * (g + 1) + g) * p.n_tiles, rp.mk};
    if (staged) {
      for (int c = threadIdx.x; c < p.n_tiles; c += kLmTailThreads) sm_mass[c] = pm(c);
      __syncthreads();
      const BlockMassScan bs = block_scan_masses(sm_mass, p.n_tiles, s_w);
      F2 local;
      const int chunk = block_pick_tile(sm_mass, bs, f2_mul_f(bs.Z, p.u_resample[b]), &local, s_pi, &s_ploc);
      if (threadIdx.x == 0) {
        s_chunk = chunk;
        s_local = local;
        s_plain = 1;
      }
    } else if (warp == 0) {
      F2 local;
      const MassScan ms = scan_masses_fn(pm, p.n_tiles);
      const int chunk = pick_chunk_fn(pm, ms, f2_mul_f(ms.Z, p.u_resample[b]), &local);
      if (lane == 0) {
        s_chunk = chunk;
        s_local = local;
        s_plain = 1;
      }
    }
    __syncthreads();
    const int chunk = s_chunk;
    const int ncol = min(kLmTileV, p.V - chunk * kLmTileV);
    const int per = (kLmTileV + gridDim.x - 1) / gridDim.x;
    const int lo = min(kLmTileV, part * per), hi = min(kLmTileV, lo + per);
    const uint4* h4 = reinterpret_cast<const uint4*>(p.hidden + static_cast<size_t>(b * (g + 1) + g) * p.H);
    for (int c = lo + warp; c < hi; c += kLmTailWarps) {
      float x = -INFINITY;
      if (c < ncol) {
        const uint4* w4 =
            reinterpret_cast<const uint4*>(p.W + (static_cast<size_t>(chunk) * kLmTileV + c) * p.H);
        x = dot_row(h4, w4, p.H / 8);
      }
      if (lane == 0) p.xsg[b * kLmTileV + c] = x;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) s_last = last_cta_arrives(&p.tail_done[b * kCounterStride], gridDim.x);
  __syncthreads();
  if (!s_last) return;

  // ---- the draw (last CTA) ----
  if (residual && staged) {  // level 1 over the residual tile masses, staged in shared memory
    for (int c = threadIdx.x; c < p.n_tiles; c += kLmTailThreads) sm_mass[c] = __ldcg(mass + c);
    __syncthreads();
    BlockMassScan bs = block_scan_masses(sm_mass, p.n_tiles, s_w);
    const bool z0 = !(bs.Z.hi > 0.f);  // uniform over the CTA
    if (z0) {
      // Z == 0 cannot happen in exact arithmetic; if rounding produces it,
      // draw from p_n itself (tile masses from its partials)
      const PartialMass pn{p.tpart + static_cast<size_t>(b * (g + 1) + s.n) * p.n_tiles, rp.mk};
      for (int c = threadIdx.x; c < p.n_tiles; c += kLmTailThreads) sm_mass[c] = pn(c);
      __syncthreads();
      bs = block_scan_masses(sm_mass, p.n_tiles, s_w);
    }
    F2 local;
    const int chunk = block_pick_tile(sm_mass, bs, f2_mul_f(bs.Z, p.u_resample[b]), &local, s_pi, &s_ploc);
    if (threadIdx.x == 0) {
      s_chunk = chunk;
      s_local = local;
      s_plain = z0;
    }
  } else if (residual && warp == 0) {  // level 1 over the residual tile masses in global memory
    bool plain = false;
    MassScan ms = scan_masses(mass, p.n_tiles);
    if (!(ms.Z.hi > 0.f)) {
      masses_from_partials(p.tpart + static_cast<size_t>(b * (g + 1) + s.n) * p.n_tiles, rp.mk, mass,
                           p.n_tiles);
      ms = scan_masses(mass, p.n_tiles);
      plain = true;
    }
    F2 local;
    const int chunk = pick_chunk(mass, ms, f2_mul_f(ms.Z, p.u_resample[b]), &local);
    if (lane == 0) {
      s_chunk = chunk;
      s_local = local;
      s_plain = plain;
    }
  }
  __syncthreads();
  const int chunk = s_chunk;
  const bool plain = s_plain;
  const int ncol = min(kLmTileV, p.V - chunk * kLmTileV);
  // the chosen tile's target logits: the stored row n, or the bonus row's recomputed tile
  if (residual) {
    const float* lp = p.logits + (static_cast<size_t>(b) * g + s.n) * p.V + static_cast<size_t>(chunk) * kLmTileV;
    for (int c = threadIdx.x; c < kLmTileV; c += kLmTailThreads) xs[c] = (c < ncol) ? __ldcg(lp + c) : -INFINITY;
  } else {
    for (int c = threadIdx.x; c < kLmTileV; c += kLmTailThreads) xs[c] = __ldcg(p.xsg + b * kLmTileV + c);
  }
  __syncthreads();
  if (warp != 0) return;

  // ---- level 2: the entry inside the tile; lane l holds entries 4l..4l+3 ----
  const F2 local = s_local;
  const WeightFn fw = plain ? make_weight(rp, rq, false, s.ks) : f;
  float xq[4] = {0.f, 0.f, 0.f, 0.f};
  if (!plain && 4 * lane < ncol)
    load_bf16x4(p.draft + (static_cast<size_t>(b) * g + s.n) * p.V + static_cast<size_t>(chunk) * kLmTileV + 4 * lane,
                xq);
  float w[4];
  F2 my = f2_from(0.f);
  int last_nz = -1;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = 4 * lane + k;
    w[k] = (e < ncol) ? fw(xs[e], xq[k]) : 0.f;
    my = f2_add(my, f2_from(w[k]));
    if (w[k] > 0.f) last_nz = e;
  }
  const F2 cincl = warp_scan_incl(my);
  const unsigned cover = __ballot_sync(0xffffffffu, f2_gt(cincl, local));
  int tok = -1;
  if (cover) {
    const int L = __ffs(cover) - 1;
    if (lane == L) {
      F2 run = f2_sub(cincl, my);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        run = f2_add(run, f2_from(w[k]));
        if (tok < 0 && f2_gt(run, local)) tok = 4 * lane + k;
      }
      if (tok < 0) tok = last_nz;  // rounding inside the lane
    }
    tok = __shfl_sync(0xffffffffu, tok, L);
  }
  if (tok < 0) {  // beyond the tile total: its last nonzero entry
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) last_nz = max(last_nz, __shfl_xor_sync(0xffffffffu, last_nz, off));
    tok = last_nz < 0 ? 0 : last_nz;
  }
  if (lane == 0) p.dp.out_tokens[b * (g + 1) + s.n] = chunk * kLmTileV + tok;
}

}  // namespace specv
