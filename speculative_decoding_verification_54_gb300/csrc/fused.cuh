// fused.cuh — the whole verify step of spec_verify_sample / spec_verify_greedy
// in one persistent launch.
//
// The step is the rejection-sampling verification of "Gemma 4 Multi-Token
// Prediction (MTP) 深度解析" §2.2 and "自投机解码：层跳过与拒绝采样实现大模型推理加速"
// §3.1-§3.2: per sequence, the temperature softmax of every target and draft
// row, the acceptance walk to the first rejection n, and a draw of position n
// from max(0, p_n - q_n) (or from p_gamma when every draft passed: "第 8 章
// 投机解码：一次前向，验证好几个字", 多出来的那一个 token 从哪来).  All of the HBM time
// is the one pass over the logits; everything after it is a chain of small
// dependent steps per sequence.  Run as separate launches, that chain waits for
// the whole pass.  Here it runs inside the pass: a sequence whose rows are
// complete is decided and drawn while the rows of later sequences still stream.
//
// Work list.  Every warp walks a fixed list of items, item i = warp + k*warps
// (round-robin, so the GPU streams the list front to back):
//   phase 1, unit b (b = 0..B-1): the chunks of rows p_0, q_0, ..., p_{g-1},
//     q_{g-1} of sequence b (stream items), then, from unit `lag` on, the
//     residual-mass items of sequence b - lag;
//   phase 2, `lag` units: the chunks of row p_gamma of a share of the
//     sequences, then the residual-mass items of one of the last `lag`
//     sequences.
// Row p_gamma only matters for the bonus token, so it streams last: by then
// most sequences are decided and drawn, and only the bonus draws remain.
//
// Who does what (no CTA ever waits for another one's progress, except the
// bounded, optional wait of a residual-mass item):
//   stream item   row chunk -> partial {max, sum, argmax, scaled max}; the
//                 warp that brings the row's chunk counter to cpr folds the row
//                 (RowStat) — the "last arriver" of the row;
//   row fold      the last phase-1 row of a sequence to be folded decides the
//                 sequence (first rejection n, emitted drafts, debug rows) and
//                 publishes its residual chunks; row p_gamma's fold writes its
//                 debug row; both then arrive at the sequence's join;
//   join          the second of {decision, p_gamma fold}: the greedy bonus
//                 (argmax of row gamma) or the sampled bonus draw from p_gamma;
//   mass item     waits (bounded) for the decision, claims one residual chunk
//                 (an epoch-tagged 64-bit counter), computes its mass of
//                 max(0, p_n - q_n) and checks in; the last of the cpr items
//                 and the decider to check in claims whatever is left (so a
//                 chunk whose item gave up waiting is never lost); the warp
//                 that completes the cpr-th mass draws the token.
// Every counter is reset by its last arriver, so the workspace is ready for the
// next call; the residual claim counter carries the call's epoch instead
// (another warp may still read it after the draw).
#pragma once

#include <cfloat>
#include <climits>

#include "common.cuh"
#include "decide.cuh"
#include "rowstats.cuh"
#include "sample.cuh"

namespace specv {

constexpr int kFusedWarps = 16;
constexpr int kFusedThreads = kFusedWarps * 32;
// How long a residual-mass item waits for its sequence's decision before it
// leaves its chunk to the cleaner (SM clock cycles, ~8 us).
constexpr long long kMassWaitCycles = 16000;
constexpr int kRowCntStride = 8;  // one 32-byte sector per row counter

// Synchronisation words of one sequence, one 128-byte line.
struct SeqSync {
  unsigned long long claim;  // (epoch << 32) | next residual chunk to hand out
  int pad0[14];
  int mass_done;  // residual chunk masses written
  int pad1[7];
  int rows_done;  // phase-1 rows folded
  int join;       // arrivals of {decision, row-gamma fold}
  int checkin;    // residual-mass items (and the decider) done claiming
  int pad2[5];
};
static_assert(sizeof(SeqSync) == 128, "one line per sequence");

struct FusedParams {
  const void* target;        // [B, gamma+1, V]
  const void* draft;         // [B, gamma, V]; nullptr: greedy entry point
  const int32_t* draft_tokens;
  const float* temperature;  // [B]; nullptr: every sequence greedy
  const float* u_accept;     // [B, gamma]
  const float* u_resample;   // [B]
  int32_t* out_tokens;
  int32_t* out_num;
  float* out_debug;          // [B, gamma+1, 4] or nullptr
  float4* partials;          // [B*S*cpr], S = 2*gamma+1 row slots per sequence
  RowStat* rowstat;          // [B*S]
  SeqState* seq;             // [B]
  float* mass;               // [B*cpr] residual chunk masses
  int* row_cnt;              // [B*S*kRowCntStride]
  SeqSync* sync;             // [B]
  WsHeader* header;          // status, epoch, CTA exit counter
  int B, gamma, V, CE, cpr;
  int lag;                   // residual items of sequence b follow phase-1 unit b + lag
  unsigned U1;               // stream items of a phase-1 unit: 2*gamma*cpr
  unsigned E1;               // items of phase 1
  unsigned N;                // items in all
};

enum WorkKind { kWorkNone = 0, kWorkStream = 1, kWorkMass = 2 };
struct Work {
  int kind, b, slot, c;
};

__device__ __forceinline__ bool fused_greedy(const FusedParams& p, int b) {
  return seq_is_greedy(p.temperature, b);
}

// Item i of the list (see the header); dead items (draft rows and residual
// items of greedy sequences) come back as kWorkNone with live = false.
__device__ __forceinline__ bool decode_work(const FusedParams& p, unsigned i, Work& w) {
  const unsigned M = static_cast<unsigned>(p.cpr);
  const unsigned K = static_cast<unsigned>(p.lag);
  unsigned off;
  if (i < p.E1) {
    unsigned u;
    if (i < K * p.U1) {
      u = i / p.U1;
      off = i - u * p.U1;
    } else {
      const unsigned i2 = i - K * p.U1, sz = p.U1 + M;
      const unsigned q = i2 / sz;
      u = K + q;
      off = i2 - q * sz;
    }
    if (off < p.U1) {
      const unsigned r = off / M;
      w.c = static_cast<int>(off - r * M);
      w.b = static_cast<int>(u);
      const int j = static_cast<int>(r >> 1);
      const bool is_draft = r & 1u;
      w.slot = is_draft ? p.gamma + 1 + j : j;
      w.kind = kWorkStream;
      return !(is_draft && fused_greedy(p, w.b));
    }
    w.b = static_cast<int>(u - K);
    w.kind = kWorkMass;
    w.c = static_cast<int>(off - p.U1);
    w.slot = 0;
    return !fused_greedy(p, w.b);
  }
  // phase 2: unit g holds the p_gamma rows of sequences [g*B/K, (g+1)*B/K)
  // and then the residual items of sequence B - K + g
  const unsigned i2 = i - p.E1, B = static_cast<unsigned>(p.B);
  unsigned g = 0, s0 = 0, s1 = B / K;  // sequences of unit g: [s0, s1)
  unsigned start = 0;                   // first item of unit g
  while (g + 1 < K) {
    const unsigned nstart = start + (s1 - s0) * M + M;
    if (i2 < nstart) break;
    start = nstart;
    ++g;
    s0 = s1;
    s1 = static_cast<unsigned>((static_cast<unsigned long long>(g + 1) * B) / K);
  }
  off = i2 - start;
  if (off < (s1 - s0) * M) {
    const unsigned r = off / M;
    w.b = static_cast<int>(s0 + r);
    w.c = static_cast<int>(off - r * M);
    w.slot = p.gamma;
    w.kind = kWorkStream;
    return true;
  }
  w.b = static_cast<int>(B - K + g);
  w.c = static_cast<int>(off - (s1 - s0) * M);
  w.slot = 0;
  w.kind = kWorkMass;
  return !fused_greedy(p, w.b);
}

// The bounds-checked build's check of a decoded item: sequence, row slot and
// chunk inside their extents (the chunk's first entry inside the row).
__device__ __forceinline__ bool work_in_bounds(const FusedParams& p, const Work& w) {
  if constexpr (!kCheckBounds) return true;
  const bool ok = w.b >= 0 && w.b < p.B && w.slot >= 0 && w.slot <= 2 * p.gamma && w.c >= 0 && w.c < p.cpr &&
                  static_cast<long long>(w.c) * p.CE < p.V;
  return in_bounds(ok, &p.header->status);
}

// The next live item of this warp at or after *i (stride nw); *i moves past it.
__device__ __forceinline__ Work next_work(const FusedParams& p, unsigned* i, unsigned nw) {
  Work w;
  while (*i < p.N) {
    const bool live = decode_work(p, *i, w);
    *i += nw;
    if (live && work_in_bounds(p, w)) return w;
  }
  w.kind = kWorkNone;
  w.b = w.slot = w.c = 0;
  return w;
}

// --- memory-model helpers (device scope) -----------------------------------
__device__ __forceinline__ int atom_add_acq_rel(int* a, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long atom_add_u64(unsigned long long* a, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(a), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ void atom_exch_release_u64(unsigned long long* a, unsigned long long v) {
  asm volatile("{\n\t.reg .b64 t;\n\tatom.release.gpu.global.exch.b64 t, [%0], %1;\n\t}" ::"l"(a), "l"(v)
               : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed(int* a, int v) {
  asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_u32(unsigned* a, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* a) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

// The caller's lane 0 arrives on *cnt; true in every lane of the warp for the
// arrival that makes the count reach `last_count` (which then resets it).
__device__ __forceinline__ bool warp_arrive_last(int* cnt, int last_count) {
  const int lane = threadIdx.x & 31;
  int is_last = 0;
  if (lane == 0) {
    const int old = atom_add_acq_rel(cnt, 1);
    is_last = (old == last_count - 1);
    if (is_last) st_relaxed(cnt, 0);
  }
  is_last = __shfl_sync(0xffffffffu, is_last, 0);
  __syncwarp();  // order lane 0's acquire before the other lanes' reads
  return is_last != 0;
}

// Streaming 16-byte load, kept in program order relative to the counters'
// atomics (the next item's loads are issued before the previous item's
// arrival so their latency overlaps it).
__device__ __forceinline__ uint4 ld_stream_ordered(const uint4* a) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(a));
  return r;
}

template <typename T>
__device__ __forceinline__ const uint8_t* fused_row(const FusedParams& p, int b, int t) {
  if (t <= p.gamma)
    return reinterpret_cast<const uint8_t*>(p.target) +
           (static_cast<size_t>(b) * (p.gamma + 1) + t) * p.V * sizeof(T);
  return reinterpret_cast<const uint8_t*>(p.draft) +
         (static_cast<size_t>(b) * p.gamma + (t - p.gamma - 1)) * p.V * sizeof(T);
}

template <typename T>
__device__ __forceinline__ void issue_loads(const FusedParams& p, const Work& w, uint4 (&v)[kVecPerLane]) {
  const int lane = threadIdx.x & 31;
  const uint4* src = reinterpret_cast<const uint4*>(fused_row<T>(p, w.b, w.slot) +
                                                    static_cast<size_t>(w.c) * p.CE * sizeof(T));
  const int nvec = min(p.CE, p.V - w.c * p.CE) / Elt<T>::kPerVec;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    const int k = lane + 32 * j;
    v[j] = (k < nvec) ? ld_stream_ordered(src + k) : neg_inf_vec<T>();
  }
}

// ---------------------------------------------------------------------------
// the draw, warp-wide (inverse CDF in ascending vocabulary order)
// ---------------------------------------------------------------------------
// Level 2 inside one chunk: lane l owns the chunk's vectors [8l, 8l+8) (a
// contiguous run, so lane order is vocabulary order); each vector's weights
// are summed in fp32, the vector sums run as two-float sums.  The vectors
// come in two halves of four (registers); the lane holding the entry reloads
// its vector for the walk.
template <typename T>
__device__ __forceinline__ float vec_weights(const uint4& a, const uint4& q, const WeightFn& f, int base,
                                             int* last_nz) {
  constexpr int P = Elt<T>::kPerVec;
  float xp[P], xq[P];
  Elt<T>::unpack(a, xp);
  Elt<T>::unpack(q, xq);
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < P; ++k) {
    const float wk = f(xp[k], xq[k]);
    s += wk;
    if (wk > 0.f) *last_nz = base + k;
  }
  return s;
}

template <typename T>
__device__ __forceinline__ int draw_in_chunk(const uint4* vp, const uint4* vq, int nvec, const WeightFn& f,
                                             bool residual, F2 local) {
  constexpr int P = Elt<T>::kPerVec;
  constexpr int H = kVecPerLane / 2;
  const int lane = threadIdx.x & 31;
  float vs[kVecPerLane];
  F2 mine = f2_from(0.f);
  int last_nz = -1;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 a[H], q[H];
#pragma unroll
    for (int j = 0; j < H; ++j) {
      const int k = lane * kVecPerLane + h * H + j;
      a[j] = (k < nvec) ? __ldg(vp + k) : neg_inf_vec<T>();
      q[j] = (residual && k < nvec) ? __ldg(vq + k) : neg_inf_vec<T>();
    }
#pragma unroll
    for (int j = 0; j < H; ++j) {
      const int jj = h * H + j;
      vs[jj] = vec_weights<T>(a[j], q[j], f, (lane * kVecPerLane + jj) * P, &last_nz);
      mine = f2_add(mine, f2_from(vs[jj]));
    }
  }
  const F2 incl = warp_scan_incl(mine);
  const unsigned over = __ballot_sync(0xffffffffu, f2_gt(incl, local));
  int tok = -1;
  if (over) {
    const int L = __ffs(over) - 1;
    if (lane == L) {
      F2 run = f2_sub(incl, mine);
      int jv = -1;
#pragma unroll
      for (int j = 0; j < kVecPerLane; ++j) {
        const F2 nxt = f2_add(run, f2_from(vs[j]));
        if (jv < 0 && f2_gt(nxt, local)) jv = j;
        if (jv < 0) run = nxt;
      }
      if (jv >= 0) {
        // the entry inside vector jv: its weights again (bitwise the same)
        const int k = lane * kVecPerLane + jv;
        const uint4 a = __ldg(vp + k);
        const uint4 q = residual ? __ldg(vq + k) : neg_inf_vec<T>();
        float xp[P], xq[P];
        Elt<T>::unpack(a, xp);
        Elt<T>::unpack(q, xq);
#pragma unroll
        for (int e = 0; e < P; ++e) {
          run = f2_add(run, f2_from(f(xp[e], xq[e])));
          if (tok < 0 && f2_gt(run, local)) tok = k * P + e;
        }
      }
      if (tok < 0) tok = -2;  // rounding inside the lane: fall back below
    }
    tok = __shfl_sync(0xffffffffu, tok, L);
  }
  if (tok < 0) {  // beyond the chunk total, or rounding: the chunk's last nonzero entry
    int m = last_nz;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
    tok = max(m, 0);
  }
  return tok;
}

// Draw position n of sequence b (s: its decision) and write the token.
// residual: level 1 runs over the residual chunk masses in p.mass; otherwise
// (bonus) over the masses of row gamma taken from its partials.
template <typename T>
__device__ __noinline__ void fused_draw(const FusedParams& p, int b, SeqState s, bool residual) {
  const int lane = threadIdx.x & 31;
  const int g = p.gamma, S = 2 * g + 1;
  if (!in_bounds(s.n >= 0 && s.n <= g && (!residual || s.n < g), &p.header->status)) return;
  const float u = p.u_resample[b];
  const RowStat* rs = p.rowstat + static_cast<size_t>(b) * S;
  int rowp = residual ? s.n : g;
  RowStat rp = ld_rowstat(rs + rowp);
  RowStat rq = residual ? ld_rowstat(rs + g + 1 + s.n) : rp;
  F2 local;
  int chunk;
  if (residual) {
    const GlobalMass gm{p.mass + static_cast<size_t>(b) * p.cpr};
    MassScan ms = scan_masses_fn(gm, p.cpr);
    if (ms.Z.hi > 0.f) {
      chunk = pick_chunk_fn(gm, ms, f2_mul_f(ms.Z, u), &local);
    } else {
      // Z == 0 cannot happen in exact arithmetic; if rounding produces it,
      // draw from p_n itself (chunk masses from its partials)
      residual = false;
      const PartialMass pn{p.partials + (static_cast<size_t>(b) * S + rowp) * p.cpr, rp.mk};
      ms = scan_masses_fn(pn, p.cpr);
      chunk = pick_chunk_fn(pn, ms, f2_mul_f(ms.Z, u), &local);
    }
  } else {
    const PartialMass pg{p.partials + (static_cast<size_t>(b) * S + rowp) * p.cpr, rp.mk};
    const MassScan ms = scan_masses_fn(pg, p.cpr);
    chunk = pick_chunk_fn(pg, ms, f2_mul_f(ms.Z, u), &local);
  }
  if (!in_bounds(chunk >= 0 && chunk < p.cpr, &p.header->status)) return;
  const WeightFn f = make_weight(rp, rq, residual, s.ks);
  const uint4* vp = chunk_vec<T>(p.target, static_cast<size_t>(b) * (g + 1) + rowp, p.V, chunk, p.CE);
  const uint4* vq =
      residual ? chunk_vec<T>(p.draft, static_cast<size_t>(b) * g + s.n, p.V, chunk, p.CE) : vp;
  const int nvec = min(p.CE, p.V - chunk * p.CE) / Elt<T>::kPerVec;
  const int tok = draw_in_chunk<T>(vp, vq, nvec, f, residual, local);
  if (lane == 0 && in_bounds(tok >= 0 && tok < nvec * Elt<T>::kPerVec, &p.header->status))
    p.out_tokens[b * (g + 1) + s.n] = chunk * p.CE + tok;
}

// ---------------------------------------------------------------------------
// residual masses: claims, the cleaner
// ---------------------------------------------------------------------------
// Mass of max(0, p_n - q_n) over chunk c, written to p.mass; the warp that
// completes the cpr-th mass draws.
template <typename T>
__device__ __noinline__ void fused_chunk(const FusedParams& p, int b, int c) {
  constexpr int P = Elt<T>::kPerVec;
  const int lane = threadIdx.x & 31;
  const int g = p.gamma, S = 2 * g + 1;
  const SeqState s = ld_seqstate(p.seq + b);
  if (!in_bounds(s.n >= 0 && s.n < g && c >= 0 && c < p.cpr, &p.header->status)) return;
  const RowStat* rs = p.rowstat + static_cast<size_t>(b) * S;
  const WeightFn f = make_weight(ld_rowstat(rs + s.n), ld_rowstat(rs + g + 1 + s.n), true, s.ks);
  const uint4* vp = chunk_vec<T>(p.target, static_cast<size_t>(b) * (g + 1) + s.n, p.V, c, p.CE);
  const uint4* vq = chunk_vec<T>(p.draft, static_cast<size_t>(b) * g + s.n, p.V, c, p.CE);
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
  acc = warp_sum(acc);
  if (lane == 0) p.mass[static_cast<size_t>(b) * p.cpr + c] = acc;
  if (warp_arrive_last(&p.sync[b].mass_done, p.cpr)) fused_draw<T>(p, b, s, true);
}

// One claim on sequence b's residual chunks: the chunk index, or -1 when none
// is left.
__device__ __forceinline__ int claim_chunk(const FusedParams& p, int b) {
  const int lane = threadIdx.x & 31;
  int c = -1;
  if (lane == 0) {
    const unsigned long long old = atom_add_u64(&p.sync[b].claim, 1ull);
    const unsigned next = static_cast<unsigned>(old & 0xffffffffull);
    if (next < static_cast<unsigned>(p.cpr)) c = static_cast<int>(next);
  }
  return __shfl_sync(0xffffffffu, c, 0);
}

// Claims until none is left (the last to check in; the claim word is already
// published for this call).
template <typename T>
__device__ __noinline__ void fused_cleaner(const FusedParams& p, int b) {
  for (int c = claim_chunk(p, b); c >= 0; c = claim_chunk(p, b)) fused_chunk<T>(p, b, c);
}

// After the last of the cpr residual items and the decider: check in.
template <typename T>
__device__ __forceinline__ void fused_checkin(const FusedParams& p, int b) {
  if (warp_arrive_last(&p.sync[b].checkin, p.cpr + 1)) fused_cleaner<T>(p, b);
}

// A residual-mass item of sequence b (sampling): wait (bounded) until the
// decision is published for this call, claim one chunk, check in.
template <typename T>
__device__ __noinline__ void fused_mass_item(const FusedParams& p, int b, unsigned epoch) {
  const int lane = threadIdx.x & 31;
  int seen = 0;
  if (lane == 0) {
    const unsigned long long* w = &p.sync[b].claim;
    long long t0 = -1;
    while (true) {
      if (static_cast<unsigned>(ld_acquire_u64(w) >> 32) == epoch) {
        seen = 1;
        break;
      }
      const long long t = clock64();
      if (t0 < 0) t0 = t;
      if (t - t0 > kMassWaitCycles) break;
      __nanosleep(64);
    }
  }
  seen = __shfl_sync(0xffffffffu, seen, 0);
  __syncwarp();
  if (seen) {
    const int c = claim_chunk(p, b);
    if (c >= 0) fused_chunk<T>(p, b, c);
  }
  fused_checkin<T>(p, b);
}

// ---------------------------------------------------------------------------
// the join of a sequence: decision + row gamma
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ void fused_join(const FusedParams& p, int b) {
  if (!warp_arrive_last(&p.sync[b].join, 2)) return;
  const SeqState s = ld_seqstate(p.seq + b);
  const int g = p.gamma;
  if (!in_bounds(s.n >= 0 && s.n <= g, &p.header->status)) return;
  if (s.mode == kModeGreedy) {
    if (s.n == g && (threadIdx.x & 31) == 0)
      p.out_tokens[b * (g + 1) + g] = ld_rowstat(p.rowstat + static_cast<size_t>(b) * (2 * g + 1) + g).argmax;
  } else if (s.mode == kModeBonus) {
    fused_draw<T>(p, b, s, false);
  }
}

// ---------------------------------------------------------------------------
// the decision (last phase-1 row of a sequence)
// ---------------------------------------------------------------------------
template <typename T>
__device__ __noinline__ void fused_decide(const FusedParams& p, int b, unsigned epoch) {
  const int lane = threadIdx.x & 31;
  const int g = p.gamma, S = 2 * g + 1;
  const bool greedy = fused_greedy(p, b);
  const RowStat* rs = p.rowstat + static_cast<size_t>(b) * S;
  DecideParams dp;
  dp.target = p.target;
  dp.draft = p.draft;
  dp.draft_tokens = p.draft_tokens;
  dp.temperature = p.temperature;
  dp.u_accept = p.u_accept;
  dp.out_tokens = p.out_tokens;
  dp.out_num = p.out_num;
  dp.out_debug = p.out_debug;
  dp.status = &p.header->status;
  dp.gamma = g;
  dp.V = p.V;
  const DecideIn in = prefetch_decide<T>(dp, b, greedy);
  const float ks = greedy ? 0.f : kLog2e / p.temperature[b];
  const int d = in.d;
  bool acc = false;
  float lp = 0.f, lq = 0.f;
  RowStat rp = {}, rq = {};
  if (lane < g) {
    rp = ld_rowstat(rs + lane);
    const bool valid = d >= 0 && d < p.V;
    if (!valid) atomicOr(&p.header->status, kStatusBadToken);
    if (valid) {
      if (greedy) {
        acc = (d == rp.argmax);
      } else {
        rq = ld_rowstat(rs + g + 1 + lane);
        lp = fmaf(in.xp, ks, -rp.mk) - rp.lse2;  // log2 p(d), log2 q(d) (debug output)
        lq = fmaf(in.xq, ks, -rq.mk) - rq.lse2;
        // log2 of the ratio from three small differences
        const float t = (in.xp - in.xq) * ks - (rp.mk - rq.mk) - (rp.lse2 - rq.lse2);
        const float rho = (in.xq == -INFINITY) ? INFINITY : ex2(t);  // q(d) == 0: accept
        acc = in.u < rho;
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
    else if (lane == n && greedy && n < g) tok = rp.argmax;  // the replacement
    // position n of a sampled sequence (and the greedy bonus) is written by
    // the draw (the join) after this store
    p.out_tokens[b * (g + 1) + lane] = tok;
  }
  if (p.out_debug != nullptr && lane < g) {
    constexpr float kLn2 = 0.6931471805599453f;
    float4 dbg;
    if (greedy) {
      const float nan = __int_as_float(0x7fc00000);
      dbg = make_float4(nan, nan, nan, nan);
    } else {
      dbg = make_float4(ex2(lp), ex2(lq), (rp.mk + rp.lse2) * kLn2, (rq.mk + rq.lse2) * kLn2);
    }
    reinterpret_cast<float4*>(p.out_debug)[b * (g + 1) + lane] = dbg;
  }
  __syncwarp();  // every lane's stores precede lane 0's release below
  if (lane == 0) {
    p.out_num[b] = n;
    SeqState st;
    st.n = n;
    st.mode = mode;
    st.ks = ks;
    st.pad = 0;
    st_seqstate(p.seq + b, st);
    if (!greedy) {
      // publish the residual chunks for this call (none unless residual)
      const unsigned long long first = (mode == kModeResidual) ? 0ull : static_cast<unsigned long long>(p.cpr);
      atom_exch_release_u64(&p.sync[b].claim, (static_cast<unsigned long long>(epoch) << 32) | first);
    }
  }
  __syncwarp();
  if (!greedy) fused_checkin<T>(p, b);
  fused_join<T>(p, b);
}

// The warp that completed row slot t of sequence b: fold it, then the chains.
template <typename T>
__device__ __noinline__ void fused_row_done(const FusedParams& p, int b, int t, unsigned epoch) {
  const int lane = threadIdx.x & 31;
  const int g = p.gamma, S = 2 * g + 1;
  const bool greedy = fused_greedy(p, b);
  const RowStat st = combine_row<4>(p.partials + (static_cast<size_t>(b) * S + t) * p.cpr, p.cpr, !greedy);
  if (lane == 0) st_rowstat(p.rowstat + static_cast<size_t>(b) * S + t, st);
  if (t == g) {
    if (p.out_debug != nullptr && lane == 0) {
      constexpr float kLn2 = 0.6931471805599453f;
      const float nan = __int_as_float(0x7fc00000);
      reinterpret_cast<float4*>(p.out_debug)[b * (g + 1) + g] =
          greedy ? make_float4(nan, nan, nan, nan) : make_float4(0.f, 0.f, (st.mk + st.lse2) * kLn2, 0.f);
    }
    __syncwarp();
    fused_join<T>(p, b);
    return;
  }
  __syncwarp();
  if (warp_arrive_last(&p.sync[b].rows_done, greedy ? g : 2 * g)) fused_decide<T>(p, b, epoch);
}

template <typename T>
__global__ void __launch_bounds__(kFusedThreads, 2) verify_fused_kernel(const __grid_constant__ FusedParams p) {
  grid_dep_launch();  // the next call's launch may overlap this one
  grid_dep_wait();    // the workspace and the logits may come from the previous grid
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned epoch = ld_relaxed_u32(&p.header->epoch) + 1u;  // this call's epoch (never 0)
  const unsigned nw = gridDim.x * kFusedWarps;
  unsigned i = blockIdx.x * kFusedWarps + warp;
  const int S = 2 * p.gamma + 1;

  Work w = next_work(p, &i, nw);
  uint4 v[kVecPerLane];
  if (w.kind == kWorkStream) issue_loads<T>(p, w, v);
  while (w.kind != kWorkNone) {
    if (w.kind == kWorkStream) {
      const int row = w.b * S + w.slot;
      const bool full = (w.slot > p.gamma) || !fused_greedy(p, w.b);
      float4 r;
      if (full) {
        r = reduce_full<T>(v, kLog2e / p.temperature[w.b]);
      } else {
        r = reduce_argmax<T>(v, w.c * p.CE, lane);
      }
      if (lane == 0) p.partials[static_cast<size_t>(row) * p.cpr + w.c] = r;
      const Work nx = next_work(p, &i, nw);
      if (nx.kind == kWorkStream) issue_loads<T>(p, nx, v);  // in flight during the arrival
      if (warp_arrive_last(p.row_cnt + static_cast<size_t>(row) * kRowCntStride, p.cpr))
        fused_row_done<T>(p, w.b, w.slot, epoch);
      w = nx;
    } else {
      fused_mass_item<T>(p, w.b, epoch);
      w = next_work(p, &i, nw);
      if (w.kind == kWorkStream) issue_loads<T>(p, w, v);
    }
  }

  // the last CTA out publishes this call's epoch for the next call
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atom_add_acq_rel(&p.header->cta_done, 1);
    if (old == static_cast<int>(gridDim.x) - 1) {
      st_relaxed(&p.header->cta_done, 0);
      st_release_u32(&p.header->epoch, epoch);
    }
  }
}

}  // namespace specv
