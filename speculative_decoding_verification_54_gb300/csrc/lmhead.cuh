// lmhead.cuh — fused lm_head GEMM on the tcgen05 tensor cores.
//
// The target logits are l[r, x] = sum_k h[r, k] * W[x, k]: hidden states of
// the verify positions times the tied embedding ("Gemma 4 Multi-Token
// Prediction (MTP) 深度解析" §3.1: lm_head shares embed_tokens; "Gemma 4 -
// Drafter 解析", 高效 Embedder: the LM head multiplies the hidden state by the
// embedding table).  No row is read back to be reduced: the epilogue turns
// each 128-entry vocabulary tile straight into the statistics the verify step
// needs.
//
// Orientation: A = a 128-row tile of W (vocabulary entries: the MMA's M and
// the TMEM lanes), B = the hidden rows (the MMA's N: up to 256 per MMA, so 320
// rows are two chunks of 160), D[vocab, row] in TMEM (fp32).  Persistent CTAs
// walk the vocabulary tiles; per CTA:
//   warp 0     one thread streams W boxes (64 x 128, 128-byte swizzle) through
//              a ring of 16 KB stages; W comes from HBM, so this ring is deep;
//   warp 1     one thread streams the hidden chunks for the same K step
//              through a second ring (they come from L2, which answers sooner);
//   warp 2     one thread issues tcgen05.mma (M=128, N=chunk, K=16) and
//              commits each stage back to its ring, and each finished chunk to
//              the epilogue;
//   warps 3-10 two groups of four (one warp per TMEM lane quadrant); both
//              work on every accumulator chunk, group g on its 32-row groups
//              of parity g, and each warp frees the chunk's TMEM slot right
//              after its last read of it.  The accumulator rotates through
//              512/chunk TMEM slots, so the epilogue of one chunk overlaps the
//              MMAs of the next (the next tile's second chunk reuses the slot
//              of this tile's first);
//   warps 11-14 the row reducer's work for the draft rows (their chunk
//              statistics), streamed from HBM beside the GEMM, which leaves
//              most of the HBM bandwidth idle.
// The epilogue holds, per thread, one vocabulary entry's logits for 32 rows at
// a time.  Per-row statistics over the tile's 128 entries come from a warp
// reduce-scatter (shuffles) followed by a combine of the four quadrant warps
// through shared memory: raw max, mk = fl(max*ks), sum 2^(fma(l, ks, -mk)),
// argmax -- the partial the row reducer makes for logits held in memory.  The
// rows that can be rejected (positions j < gamma of sampling sequences) are
// also stored in fp32, a warp writing 32 consecutive vocabulary entries of a
// row at once: the residual max(0, p_j - q_j) needs p_j's normaliser, known
// only once the whole row is reduced.  At B=64, gamma=4, H=1536 the store
// measured 51 us of a 298 us launch, where recomputing the rows the draw
// needs (a second pass over W for 64 rows) measured 175 us.
#pragma once

#include <cfloat>
#include <cuda.h>

#include "common.cuh"
#include "rowstats.cuh"
#include "tc.cuh"

namespace specv {

constexpr int kLmTileV = 128;       // vocabulary entries per tile (MMA M, TMEM lanes)
constexpr int kLmTileK = 64;        // K per stage: one 128-byte swizzled row of bf16
constexpr int kLmMaxRows = 384;     // hidden rows per call
constexpr int kLmMaxChunk = 256;    // MMA N limit
constexpr uint32_t kLmWBytes = kLmTileV * kLmTileK * 2;  // 16 KB
constexpr int kLmMaxWStages = 6, kLmMaxHStages = 6, kLmMaxSlots = 4;
// W steps prefetched into L2 ahead of the ring (64 KB per CTA).  Measured (GEMM
// alone, B=64, H=1536, one box): 4 steps 241.6 us, 8 steps 244.0, 12 steps
// 245.7, 20 steps 276.2, 32 steps 300.6: a long lead only evicts lines.
constexpr int kLmWPrefetch = 4;
constexpr int kLmEpiGroups = 2;                                         // of four warps
constexpr int kLmRowWarp0 = 3 + 4 * kLmEpiGroups;                       // first row warp
constexpr int kLmRowWarps = 4;                                          // the draft rows' statistics
constexpr int kLmThreads = 32 * (kLmRowWarp0 + kLmRowWarps);            // 480
constexpr uint32_t kLmTmemCols = 512;

struct LmParams {
  CUtensorMap tmW;  // W [V, H] bf16, box 64 x 128
  CUtensorMap tmH;  // hidden [R, H] bf16, box 64 x nc
  int R, V, H, n_tiles, gamma;
  int nc, n_chunks, n_slots;  // chunk width (multiple of 32, <= 256), chunks per tile, TMEM slots
  int w_stages, h_stages;
  uint32_t h_bytes;           // one hidden stage: n_chunks * nc rows of 128 bytes
  const float* temperature;   // [B]
  float4* partials;           // [R][n_tiles] {M, s, argmax bits, mk}
  float* logits;              // [B, gamma, V] fp32, rows j < gamma of sampling sequences
  int* status;
  // the draft rows' chunk statistics (the row reducer's items, target rows
  // skipped), computed by the row warps beside the GEMM; rows.draft ==
  // nullptr: none
  RowStatsParams rows;
};

// Dynamic shared memory: W ring, hidden ring, the epilogue's cross-warp
// scratch (red [4][nc] f32, redI [4][nc] i32, fin [nc] float2, finM [nc] f32,
// finI [nc] i32; the groups use disjoint rows of it), then per epilogue warp a
// transpose buffer for the stored logits.
__host__ __device__ inline uint32_t lm_scratch_bytes(int nc) { return static_cast<uint32_t>(nc) * 4u * 12u; }
constexpr uint32_t kLmTransBytes = 8 * 32 * 4;  // per epilogue warp: 8 rows x 32 entries
__host__ __device__ inline uint32_t lm_smem_bytes(int w_stages, int h_stages, uint32_t h_bytes, int nc) {
  return static_cast<uint32_t>(w_stages) * kLmWBytes + static_cast<uint32_t>(h_stages) * h_bytes +
         lm_scratch_bytes(nc) + 4u * kLmEpiGroups * kLmTransBytes + 1024u;
}

// 32-byte global store (eight fp32; the address 32-byte aligned)
__device__ __forceinline__ void st_global_v8(float* q, const float4& lo, const float4& hi) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(q), "f"(lo.x), "f"(lo.y), "f"(lo.z),
               "f"(lo.w), "f"(hi.x), "f"(hi.y), "f"(hi.z), "f"(hi.w)
               : "memory");
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Warp reduce-scatter over 32 columns.  On entry lane l holds v[j] = the value
// of column j at its own vocabulary entry (index id[j]); on return v[0] (and
// id[0]) of lane l is column l's maximum over the warp's 32 entries, the
// lowest index on ties when kIdx.
template <bool kIdx>
__device__ __forceinline__ void rs_max(float (&v)[32], int (&id)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool hi = (lane & s) != 0;
#pragma unroll
    for (int j = 0; j < s; ++j) {
      const float send = hi ? v[j] : v[j + s];
      const float keep = hi ? v[j + s] : v[j];
      const float got = __shfl_xor_sync(0xffffffffu, send, s);
      if (kIdx) {
        const int isend = hi ? id[j] : id[j + s];
        const int ikeep = hi ? id[j + s] : id[j];
        const int igot = __shfl_xor_sync(0xffffffffu, isend, s);
        const bool take = got > keep || (got == keep && igot < ikeep);
        v[j] = take ? got : keep;
        id[j] = take ? igot : ikeep;
      } else {
        v[j] = fmaxf(got, keep);
      }
    }
  }
}

// The same for sums: on return v[0] of lane l is column l's sum over the warp.
__device__ __forceinline__ void rs_sum(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool hi = (lane & s) != 0;
#pragma unroll
    for (int j = 0; j < s; ++j) {
      const float send = hi ? v[j] : v[j + s];
      const float keep = hi ? v[j + s] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
}

// Per-row constants of the epilogue, filled once per CTA.
struct LmRowTables {
  float ks[kLmMaxRows];      // log2(e)/T for sampled rows, 0 otherwise
  int srow[kLmMaxRows];      // row of the stored-logits tensor, or -1
  int8_t greedy[kLmMaxRows];  // 1 for rows of greedy sequences
};

struct LmEpiScratch {
  float* red;   // [4][nc]
  int* redI;    // [4][nc]
  float2* fin;  // [nc] {ks, mk} (mk = +inf for rows without exponentials)
  float* finM;  // [nc] row maxima over the tile
  int* finI;    // [nc] their lowest vocabulary index (greedy rows), else -1
  float* tb;    // this warp's [8][32] transpose buffer
};

// One accumulator chunk (nc hidden rows x 128 vocabulary entries) of tile
// `tile`: this group of four warps (this warp: lane quadrant `quad`) takes
// the chunk's 32-row groups g0, g0 + 2, ... (the other group the rest), so
// both groups work on a chunk at once and its TMEM slot is freed sooner.
// Phase 1: per 32-row group, the warp's column maxima (and argmax where a row
// is greedy) into red/redI.  Phase 2: lane l combines the four quadrants for
// row l of each group.  Phase 3: exponentials against the row maxima, the
// stored logits, and the warp's column sums into red; each warp frees the
// TMEM slot right after its last read of the chunk.  Phase 4: the row
// partials.  The group
// loops stay rolled (the unrolled bodies overflow the instruction cache);
// what crosses phases lives in shared memory.
__device__ __forceinline__ void lm_epilogue_chunk(const LmParams& p, const LmRowTables& T, const LmEpiScratch& S,
                                                  uint32_t tacc, int tile, int c, int g0, int quad, int lane,
                                                  int bar_id, uint64_t* slot_empty) {
  const int nc = p.nc, ng = nc / 32;
  const int x = tile * kLmTileV + quad * 32 + lane;  // this lane's vocabulary entry
  const bool xv = x < p.V;
  // this group's row of phases 2 and 4: quadrant warp q takes the group's
  // q-th 32-row group (at most (ng + 1) / 2 <= 4 of them)
  const int my_g = g0 + 2 * quad;
  const int col = my_g * 32 + lane;
  const bool has_col = my_g < ng;

  // ---- phase 1 ----
#pragma unroll 1
  for (int g = g0; g < ng; g += 2) {
    float v[32];
    int id[32];
    tmem_ld32(tacc + g * 32, v);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      v[j] = xv ? v[j] : -INFINITY;
      id[j] = x;
    }
    const int rb = c * nc + g * 32;
    const bool anyg = __any_sync(0xffffffffu, rb + lane < p.R && T.greedy[rb + lane]);
    if (anyg) {
      rs_max<true>(v, id, lane);
      S.redI[quad * nc + g * 32 + lane] = id[0];
    } else {
      rs_max<false>(v, id, lane);
    }
    S.red[quad * nc + g * 32 + lane] = v[0];
  }
  named_bar(bar_id, 128);

  // ---- phase 2: the four quadrants of each of the group's rows ----
  if (has_col) {
    const int row = c * nc + col;
    const bool rv = row < p.R;
    const bool gr = rv && T.greedy[row];
    float M = S.red[col];
    int I = gr ? S.redI[col] : -1;
#pragma unroll
    for (int q = 1; q < 4; ++q) {
      const float o = S.red[q * nc + col];
      if (gr) {
        const int oi = S.redI[q * nc + col];
        if (o > M || (o == M && oi < I)) {
          M = o;
          I = oi;
        }
      } else {
        M = fmaxf(M, o);
      }
    }
    const float ks = rv ? T.ks[row] : 0.f;
    const bool sampled = ks > 0.f && M > -FLT_MAX;
    S.fin[col] = make_float2(ks, sampled ? M * ks : INFINITY);
    S.finM[col] = M;
    S.finI[col] = I;
  }
  named_bar(bar_id, 128);

  // ---- phase 3 ----
  // The slot is released right after this warp's last TMEM read of the
  // chunk (the values are in registers from then on), so the next tile's
  // MMAs do not wait for the last group's exponentials and stores.
  if (g0 >= ng) {  // no 32-row group of this chunk for this group
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(slot_empty);
  }
#pragma unroll 1
  for (int g = g0; g < ng; g += 2) {
    float v[32];
    tmem_ld32(tacc + g * 32, v);
    if (g + 2 >= ng) {  // this warp's last read of the chunk
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(slot_empty);
    }
    const int rb = c * nc + g * 32;
    const bool anys = __any_sync(0xffffffffu, S.fin[g * 32 + lane].y < INFINITY);
    const int srl = (rb + lane < p.R) ? T.srow[rb + lane] : -1;
    const unsigned stmask = __ballot_sync(0xffffffffu, srl >= 0);
    if (stmask != 0u) {
      // 8 rows at a time through the transpose buffer, so that each store
      // writes 32 bytes per lane: eight rows x 128 bytes per instruction (one
      // 32-byte store measured 259.7 us per launch against 263.5 us with two
      // of 16 bytes)
      const int x0 = tile * kLmTileV + quad * 32;
#pragma unroll
      for (int b8 = 0; b8 < 4; ++b8) {
        if (((stmask >> (8 * b8)) & 0xffu) == 0u) continue;  // warp-uniform
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) S.tb[jj * 32 + lane] = v[8 * b8 + jj];
        __syncwarp();
        {
          // lane -> row rr of the eight, entries c8..c8+7 (32-byte aligned: V
          // is a multiple of 8)
          const int rr = lane >> 2, c8 = (lane & 3) * 8;
          const int sr = __shfl_sync(0xffffffffu, srl, 8 * b8 + rr);
          const float4 lo = *reinterpret_cast<const float4*>(S.tb + rr * 32 + c8);
          const float4 hi = *reinterpret_cast<const float4*>(S.tb + rr * 32 + c8 + 4);
          if (sr >= 0 && x0 + c8 < p.V) st_global_v8(p.logits + static_cast<size_t>(sr) * p.V + x0 + c8, lo, hi);
        }
        __syncwarp();
      }
    }
    if (anys) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float2 f = S.fin[g * 32 + j];
        v[j] = xv ? ex2(fmaf(v[j], f.x, -f.y)) : 0.f;
      }
      rs_sum(v, lane);
      S.red[quad * nc + g * 32 + lane] = v[0];
    }
  }
  named_bar(bar_id, 128);

  // ---- phase 4 ----
  if (tile < p.n_tiles) {
    if (has_col) {
      const int row = c * nc + col;
      if (row < p.R) {
        const float2 f = S.fin[col];
        float s = 0.f;
        if (f.y < INFINITY) s = (S.red[col] + S.red[nc + col]) + (S.red[2 * nc + col] + S.red[3 * nc + col]);
        p.partials[static_cast<size_t>(row) * p.n_tiles + tile] =
            make_float4(S.finM[col], s, __int_as_float(S.finI[col]), f.y < INFINITY ? f.y : kNegHuge);
      }
    }
  }
  named_bar(bar_id, 128);  // scratch free for the group's next chunk
}

// kChunks: accumulator chunks per tile (1 or 2, = p.n_chunks), a compile-time
// constant so the producer and MMA threads, which run once per K step, carry
// no chunk loop or test (at one chunk of 64 rows that measured 147 us against
// 177 us with the count read at run time)
template <int kChunks>
__global__ void __launch_bounds__(kLmThreads, 1) lmhead_kernel(const __grid_constant__ LmParams p) {
  extern __shared__ __align__(1024) uint8_t lm_smem_raw[];
  uint8_t* smem = lm_smem_raw + ((1024u - (smem_u32(lm_smem_raw) & 1023u)) & 1023u);
  uint8_t* wring = smem;
  uint8_t* hring = smem + p.w_stages * kLmWBytes;
  uint8_t* scratch = hring + p.h_stages * p.h_bytes;
  __shared__ __align__(8) uint64_t wfull[kLmMaxWStages], wempty[kLmMaxWStages];
  __shared__ __align__(8) uint64_t hfull[kLmMaxHStages], hempty[kLmMaxHStages];
  __shared__ __align__(8) uint64_t sfull[kLmMaxSlots], sempty[kLmMaxSlots];
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort[kLmEpiGroups];
  __shared__ LmRowTables T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_launch();

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.w_stages; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 1);
    }
    for (int s = 0; s < p.h_stages; ++s) {
      mbar_init(&hfull[s], 1);
      mbar_init(&hempty[s], 1);
    }
    for (int s = 0; s < p.n_slots; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 4 * kLmEpiGroups);  // every epilogue warp reads every chunk
    }
    for (int g = 0; g < kLmEpiGroups; ++g) s_abort[g] = 0;
    fence_mbar_init();
  }
  // per-row constants (inputs of the call: no dependency on earlier kernels)
  for (int r = threadIdx.x; r < kLmMaxRows; r += kLmThreads) {
    float ks = 0.f;
    int srow = -1;
    int8_t gr = 0;
    if (r < p.R) {
      const int b = r / (p.gamma + 1), j = r - b * (p.gamma + 1);
      gr = seq_is_greedy(p.temperature, b) ? 1 : 0;
      if (!gr) {
        ks = kLog2e / p.temperature[b];
        if (j < p.gamma) srow = b * p.gamma + j;
      }
    }
    T.ks[r] = ks;
    T.srow[r] = srow;
    T.greedy[r] = gr;
  }
  if (warp == 2) tmem_alloc(&tmem_base, kLmTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  const int ksteps = p.H / kLmTileK;
  const int my_tiles = (p.n_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                       static_cast<int>(gridDim.x);
  const int nsteps = my_tiles * ksteps;
  if (warp == 0 || warp == 1) {
    // ---------------- producers: warp 0 the W ring, warp 1 the hidden ring ----------------
    // Stage index, phase parity, tile and K step advance incrementally: this
    // thread is on the critical path of every K step.
    if (lane == 0) {
      const bool isw = (warp == 0);
      const int nst = isw ? p.w_stages : p.h_stages;
      uint64_t* full = isw ? wfull : hfull;
      uint64_t* empty = isw ? wempty : hempty;
      uint8_t* ring = isw ? wring : hring;
      const uint32_t sbytes = isw ? kLmWBytes : p.h_bytes;
      const uint32_t cbytes = static_cast<uint32_t>(p.nc) * 128u;
      // each CTA walks K from its own offset, so the CTAs do not all read the
      // same hidden-state columns from L2 at once
      const int k0 = static_cast<int>(blockIdx.x) % ksteps;
      int s = 0, k = k0, kc = 0, tile = static_cast<int>(blockIdx.x), i = 0;
      uint32_t ph = 0;
      // W: L2 prefetch kLmWPrefetch steps ahead, so the ring's own loads hit L2
      int pk = k0, pkc = 0, ptile = tile, pi = 0;
      if (isw) {
        for (; pi < nsteps && pi < kLmWPrefetch; ++pi) {
          tma_prefetch_2d(&p.tmW, pk * kLmTileK, ptile * kLmTileV);
          if (++pk == ksteps) pk = 0;
          if (++pkc == ksteps) {
            pkc = 0;
            ptile += static_cast<int>(gridDim.x);
          }
        }
      }
      for (; i < nsteps; ++i) {
        if (i >= nst && !mbar_wait(&empty[s], ph ^ 1u, p.status, kWaitLimitCycles)) break;
        uint8_t* dst = ring + s * sbytes;
        mbar_arrive_expect_tx(&full[s], sbytes);
        if (isw) {
          tma_load_2d(dst, &p.tmW, k * kLmTileK, tile * kLmTileV, &full[s]);
          if (pi < nsteps) {
            tma_prefetch_2d(&p.tmW, pk * kLmTileK, ptile * kLmTileV);
            ++pi;
            if (++pk == ksteps) pk = 0;
            if (++pkc == ksteps) {
              pkc = 0;
              ptile += static_cast<int>(gridDim.x);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < kChunks; ++c) tma_load_2d(dst + c * cbytes, &p.tmH, k * kLmTileK, c * p.nc, &full[s]);
        }
        if (++k == ksteps) k = 0;
        if (++kc == ksteps) {
          kc = 0;
          tile += static_cast<int>(gridDim.x);
        }
        if (++s == nst) {
          s = 0;
          ph ^= 1u;
        }
      }
      // drain: the copies of the last stages land before the CTA exits
      for (int j = (i > nst ? i - nst : 0); j < i; ++j)
        mbar_wait(&full[j % nst], (j / nst) & 1, p.status, kWaitLimitCycles);
    }
  } else if (warp == 2) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kLmTileV, p.nc);
      const uint32_t cbytes = static_cast<uint32_t>(p.nc) * 128u;
      const uint64_t wdesc0 = smem_desc_k128(smem_u32(wring)), hdesc0 = smem_desc_k128(smem_u32(hring));
      constexpr bool two = kChunks > 1;
      int sw = 0, sh = 0, su = 0, u = 0;
      uint32_t pw = 0, phh = 0, pu = 0;
      bool ok = true;
      for (int t = 0; t < my_tiles && ok; ++t) {
        uint32_t dcol[2];
        int dslot[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // n_chunks <= 2
          dslot[c] = su;
          dcol[c] = tmem + static_cast<uint32_t>(su * p.nc);
          if (c < kChunks) {
            if (u >= p.n_slots && !mbar_wait(&sempty[su], pu ^ 1u, p.status, kWaitLimitCycles)) ok = false;
            ++u;
            if (++su == p.n_slots) {
              su = 0;
              pu ^= 1u;
            }
          }
        }
        if (!ok) break;
        tc_fence_after();
        for (int k = 0; k < ksteps; ++k) {
          if (!mbar_wait(&wfull[sw], pw, p.status, kWaitLimitCycles) ||
              !mbar_wait(&hfull[sh], phh, p.status, kWaitLimitCycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptors of the stage; a K=16 slice is 32 bytes further, +2 in
          // the start-address field (16-byte units)
          const uint64_t ad = wdesc0 + static_cast<uint64_t>(sw) * (kLmWBytes >> 4);
          const uint64_t bd = hdesc0 + static_cast<uint64_t>(sh) * (p.h_bytes >> 4);
#pragma unroll
          for (int kk = 0; kk < kLmTileK / 16; ++kk) {
            tc_mma(dcol[0], ad + 2 * kk, bd + 2 * kk, idesc, k > 0 || kk > 0);
            if (two) tc_mma(dcol[1], ad + 2 * kk, bd + (cbytes >> 4) + 2 * kk, idesc, k > 0 || kk > 0);
          }
          tc_commit(&wempty[sw]);  // the stages are free once these MMAs have read them
          tc_commit(&hempty[sh]);
          if (++sw == p.w_stages) {
            sw = 0;
            pw ^= 1u;
          }
          if (++sh == p.h_stages) {
            sh = 0;
            phh ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&sfull[dslot[0]]);
        if (two) tc_commit(&sfull[dslot[1]]);
      }
    }
  } else if (warp < kLmRowWarp0) {
    // ---------------- epilogue: warps 3..10, two groups of four ----------------
    const int e = warp - 3, grp = e >> 2, quad = warp & 3;
    LmEpiScratch S;
    // one scratch for both groups: group g always takes the 32-row groups of
    // parity g, so the two never touch the same rows of it
    uint8_t* sc = scratch;
    S.red = reinterpret_cast<float*>(sc);
    S.redI = reinterpret_cast<int*>(sc + 16 * p.nc);
    S.fin = reinterpret_cast<float2*>(sc + 32 * p.nc);
    S.finM = reinterpret_cast<float*>(sc + 40 * p.nc);
    S.finI = reinterpret_cast<int*>(sc + 44 * p.nc);
    S.tb = reinterpret_cast<float*>(scratch + lm_scratch_bytes(p.nc) + e * kLmTransBytes);
    const int units = my_tiles * kChunks;
    for (int u = 0; u < units; ++u) {
      const int slot = u % p.n_slots;
      const bool got = __all_sync(0xffffffffu, mbar_wait(&sfull[slot], (u / p.n_slots) & 1, p.status,
                                                         kWaitLimitCycles));
      if (!got && lane == 0) s_abort[grp] = 1;
      named_bar(1 + grp, 128);
      if (s_abort[grp]) break;  // uniform over the group
      tc_fence_after();
      const int t = u / kChunks, c = u % kChunks;
      const int tile = static_cast<int>(blockIdx.x) + t * static_cast<int>(gridDim.x);
      const uint32_t tacc = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(slot * p.nc);
      lm_epilogue_chunk(p, T, S, tacc, tile, c, grp, quad, lane, 1 + grp, &sempty[slot]);
    }
  } else {
    // ---------------- row warps: the draft rows' chunk statistics ----------------
    // The row reducer's items (one 4 KB chunk of a draft row per warp and
    // step), dealt over the grid's row warps.  The draft logits are inputs of
    // the call, so this streaming overlaps the GEMM: it takes HBM bandwidth
    // the W stream leaves idle.
    const RowStatsParams& rp = p.rows;
    if (rp.draft != nullptr) {
      const int n_slots = rp.B * (2 * rp.gamma + 1);
      ItemIter it;
      it.init(static_cast<int>(blockIdx.x) * kLmRowWarps + (warp - kLmRowWarp0),
              static_cast<int>(gridDim.x) * kLmRowWarps, rp.cpr);
      Item d;
      while (next_live<__nv_bfloat16>(rp, it, n_slots, d)) {
        uint4 v[kVecPerLane];
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j) {
          const int k = lane + 32 * j;
          v[j] = (k < d.nvec) ? ld_stream(d.src + k) : neg_inf_vec<__nv_bfloat16>();
        }
        finish_item<__nv_bfloat16, false>(rp, d, v, lane);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, kLmTmemCols);
}

}  // namespace specv
