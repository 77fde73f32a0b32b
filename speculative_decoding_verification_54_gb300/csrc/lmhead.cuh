// lmhead.cuh — fused lm_head GEMM on the tcgen05 tensor cores.
//
// The target logits are l[r, x] = sum_k h[r, k] * W[x, k]: hidden states of
// the verify positions times the tied embedding ("Gemma 4 Multi-Token
// Prediction (MTP) 深度解析" §3.1: lm_head shares embed_tokens; "Gemma 4 -
// Drafter 解析", 高效 Embedder: the LM head multiplies the hidden state by the
// embedding table).  They are never written to memory: the epilogue turns each
// 128-entry vocabulary tile straight into the statistics the verify step needs.
//
// Orientation: A = hidden rows (up to three 128-row M-tiles, 384 rows), B = a
// 128-row tile of W, D[row, vocab] in TMEM (fp32, 128 columns per M-tile).  A
// TMEM lane is one hidden row, so each epilogue thread owns a row's logits and
// needs no cross-thread reduction.  Persistent CTAs walk the vocabulary tiles;
// per CTA:
//   warp 0    one thread issues 2-D TMA tile loads (128-byte swizzle) of A and
//             B into a 3-stage ring of 64 KB stages (full/empty mbarriers);
//   warp 1    one thread issues tcgen05.mma (M=128, N=128, K=16, bf16 -> f32)
//             and commits each stage back to its empty barrier, and the
//             finished tile to the epilogue;
//   warps 2-5 read the accumulator with tcgen05.ld and reduce it.
// The epilogue writes, per (row, tile), the partial the row reducer makes for
// logits held in memory -- raw max, mk = fl(max*ks), sum 2^(fma(l, ks, -mk)),
// argmax -- and, for the rows that can be rejected (positions j < gamma of
// sampling sequences), the tile's 128 fp32 logits: the residual
// max(0, p_j - q_j) needs p_j's normaliser, known only once the whole row is
// reduced, and storing these rows (4 bytes per entry) costs a third of
// reading W a second time.
#pragma once

#include <cfloat>
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace specv {

constexpr int kLmTileM = 128, kLmTileN = 128, kLmTileK = 64;
constexpr int kLmMaxMTiles = 3;
constexpr int kLmStages = 3;
constexpr uint32_t kLmABytes = kLmTileM * kLmTileK * 2;                      // 16 KB
constexpr uint32_t kLmBBytes = kLmTileN * kLmTileK * 2;                      // 16 KB
constexpr uint32_t kLmStageBytes = kLmMaxMTiles * kLmABytes + kLmBBytes;     // 64 KB
constexpr uint32_t kLmSmemBytes = kLmStages * kLmStageBytes + 1024;          // + alignment slack
constexpr int kLmThreads = 192;
constexpr uint32_t kLmTmemCols = 512;

struct LmParams {
  CUtensorMap tmA;  // hidden rows [R, H] bf16, box 64 x 128
  CUtensorMap tmB;  // W [V, H] bf16, box 64 x 128
  int R, n_mtiles, V, H, n_tiles, gamma;
  const float* temperature;  // [B]
  float4* partials;          // [R][n_tiles] {M, s, argmax bits, mk}
  float* logits;             // [B, gamma, V] fp32, rows j < gamma of sampling sequences
  int* status;
};

// This thread's 128 accumulator columns of one M-tile (warp-wide call).
__device__ __forceinline__ void lm_load_row(uint32_t taddr, float (&v)[kLmTileN]) {
#pragma unroll
  for (int c = 0; c < kLmTileN / 32; ++c) {
    float t[32];
    tmem_ld32(taddr + c * 32, t);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[c * 32 + i] = t[i];
  }
}

// Epilogue of row r for tile `tile` (ncol valid columns, a multiple of 8):
// the partial, and the logits themselves when `store` is non-null.
__device__ __forceinline__ void lm_epilogue_row(const LmParams& p, const float (&v)[kLmTileN], int r, int tile,
                                                int ncol, float ks, bool greedy, float* store) {
  float m = -FLT_MAX;
  int idx = -1;
#pragma unroll
  for (int c = 0; c < kLmTileN; ++c) {
    const float x = (c < ncol) ? v[c] : -INFINITY;
    const bool gt = x > m;  // strict: the lowest index keeps a tie
    m = gt ? x : m;
    idx = gt ? tile * kLmTileN + c : idx;
  }
  float s = 0.f, mk = kNegHuge;
  if (!greedy && m > -FLT_MAX) {
    mk = m * ks;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int c = 0; c < kLmTileN; c += 4) {
      s0 += (c + 0 < ncol) ? ex2(fmaf(v[c + 0], ks, -mk)) : 0.f;
      s1 += (c + 1 < ncol) ? ex2(fmaf(v[c + 1], ks, -mk)) : 0.f;
      s2 += (c + 2 < ncol) ? ex2(fmaf(v[c + 2], ks, -mk)) : 0.f;
      s3 += (c + 3 < ncol) ? ex2(fmaf(v[c + 3], ks, -mk)) : 0.f;
    }
    s = (s0 + s1) + (s2 + s3);
  }
  p.partials[static_cast<size_t>(r) * p.n_tiles + tile] = make_float4(m, s, __int_as_float(idx), mk);
  if (store != nullptr) {
    float4* dst = reinterpret_cast<float4*>(store + static_cast<size_t>(tile) * kLmTileN);
#pragma unroll
    for (int c4 = 0; c4 < kLmTileN / 4; ++c4)
      if (c4 * 4 < ncol) dst[c4] = make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
  }
}

__global__ void __launch_bounds__(kLmThreads, 1) lmhead_kernel(const __grid_constant__ LmParams p) {
  extern __shared__ __align__(1024) uint8_t lm_smem_raw[];
  uint8_t* smem = lm_smem_raw + ((1024u - (smem_u32(lm_smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t full_bar[kLmStages], empty_bar[kLmStages], tfull_bar, tempty_bar;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_launch();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLmStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&tfull_bar, 1);
    mbar_init(&tempty_bar, 4);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_base, kLmTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  const int ksteps = p.H / kLmTileK;
  const int nm = p.n_mtiles;
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint32_t bytes = nm * kLmABytes + kLmBBytes;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.n_tiles && ok; tile += gridDim.x) {
        for (int k = 0; k < ksteps; ++k, ++it) {
          const int s = it % kLmStages;
          if (it >= kLmStages &&
              !mbar_wait(&empty_bar[s], ((it / kLmStages) & 1) ^ 1, p.status, kWaitLimitCycles)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kLmStageBytes;
          mbar_arrive_expect_tx(&full_bar[s], bytes);
          for (int m = 0; m < nm; ++m)
            tma_load_2d(st + m * kLmABytes, &p.tmA, k * kLmTileK, m * kLmTileM, &full_bar[s]);
          tma_load_2d(st + kLmMaxMTiles * kLmABytes, &p.tmB, k * kLmTileK, tile * kLmTileN, &full_bar[s]);
        }
      }
      // drain: the copies of the last kLmStages stages land before exit
      for (int j = (it > kLmStages ? it - kLmStages : 0); j < it; ++j)
        mbar_wait(&full_bar[j % kLmStages], (j / kLmStages) & 1, p.status, kWaitLimitCycles);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kLmTileM, kLmTileN);
      int it = 0, tcount = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.n_tiles && ok; tile += gridDim.x, ++tcount) {
        if (tcount > 0 && !mbar_wait(&tempty_bar, (tcount - 1) & 1, p.status, kWaitLimitCycles)) break;
        tc_fence_after();
        for (int k = 0; k < ksteps; ++k, ++it) {
          const int s = it % kLmStages;
          if (!mbar_wait(&full_bar[s], (it / kLmStages) & 1, p.status, kWaitLimitCycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * kLmStageBytes);
#pragma unroll
          for (int kk = 0; kk < kLmTileK / 16; ++kk) {
            const uint64_t bdesc = smem_desc_k128(st + kLmMaxMTiles * kLmABytes + kk * 32);
            for (int m = 0; m < nm; ++m)
              tc_mma(tmem + m * kLmTileN, smem_desc_k128(st + m * kLmABytes + kk * 32), bdesc, idesc,
                     k > 0 || kk > 0);
          }
          tc_commit(&empty_bar[s]);  // the stage is free once these MMAs have read it
        }
        if (ok) tc_commit(&tfull_bar);
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5, TMEM lane quadrant warp % 4 ----------------
    const int quad = warp & 3;
    // per-row constants, hoisted out of the tile loop
    float ks[kLmMaxMTiles];
    bool greedy[kLmMaxMTiles];
    float* store[kLmMaxMTiles];
#pragma unroll
    for (int m = 0; m < kLmMaxMTiles; ++m) {
      const int r = m * kLmTileM + quad * 32 + lane;
      ks[m] = 0.f;
      greedy[m] = true;
      store[m] = nullptr;
      if (r < p.R) {
        const int b = r / (p.gamma + 1), j = r - b * (p.gamma + 1);
        greedy[m] = seq_is_greedy(p.temperature, b);
        ks[m] = greedy[m] ? 0.f : kLog2e / p.temperature[b];
        if (!greedy[m] && j < p.gamma) store[m] = p.logits + (static_cast<size_t>(b) * p.gamma + j) * p.V;
      }
    }
    int tcount = 0;
    for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x, ++tcount) {
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull_bar, tcount & 1, p.status, kWaitLimitCycles))) break;
      tc_fence_after();
      const int ncol = min(kLmTileN, p.V - tile * kLmTileN);
      const uint32_t tlane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll
      for (int m = 0; m < kLmMaxMTiles; ++m) {
        if (m < nm) {  // warp-uniform
          float v[kLmTileN];
          lm_load_row(tlane + m * kLmTileN, v);
          const int r = m * kLmTileM + quad * 32 + lane;
          if (r < p.R) lm_epilogue_row(p, v, r, tile, ncol, ks[m], greedy[m], store[m]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kLmTmemCols);
  grid_dep_wait();  // the row reducer launched before this kernel has finished too
}

}  // namespace specv
