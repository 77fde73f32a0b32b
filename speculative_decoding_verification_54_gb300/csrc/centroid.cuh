// centroid.cuh — the centroid-masked sparse draft head.
//
// "Gemma 4 Multi-Token Prediction (MTP) 深度解析" §3.4 Centroids Masking and
// "Gemma 4 - Drafter 解析", 高效 Embedder: the drafter of the small Gemma 4
// models scores clusters of tokens instead of the whole vocabulary.  The
// token embeddings are stored cluster by cluster (cluster c owns the ordered
// rows cluster_off[c] .. cluster_off[c+1]-1; ordered row i is token
// ord2tok[i]); one embedding per cluster (its centroid) scores the clusters
// against the drafter's hidden state, the top_k clusters are kept, and token
// logits are computed only for their tokens.  Four kernels, chained with
// programmatic dependent launch:
//   cluster_score_*        z[r, c] = h[r] . C[c]  (fp32 sums of bf16 products):
//                          for more than 16 hidden rows a tcgen05 GEMM (128
//                          centroids x up to 256 hidden rows per CTA, K split
//                          over up to 8 CTAs); for fewer, CUDA cores (each
//                          warp holds one centroid, the CTA stages
//                          kHeadRowBlock hidden rows in shared memory)
//   cluster_topk_kernel    one CTA per row: adds the K-split partial scores in
//                          order, radix select of the top_k scores
//                          (the lowest index first among equal scores) and
//                          the selected clusters' candidate offsets
//   cand_logit_kernel      grid (top_k, R): one CTA per selected cluster, one
//                          warp per token row, writes (token, logit) unsorted
//   cand_sort_kernel       one CTA per row: orders the candidates by token id
//                          (the order the sparse verification searches in):
//                          ranks from a bitmap of the row's tokens
// The bulk of the bytes is the gathered embedding rows (top_k clusters of
// about V / n_clusters rows of 2H bytes per hidden row): HBM/L2 bound.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "tc.cuh"
#include "topkp.cuh"

namespace specv {

constexpr int kHeadThreads = 512;  // tk_sort_desc assumes 512-thread CTAs
constexpr int kHeadWarps = kHeadThreads / 32;
constexpr int kHeadRowBlock = 4;       // hidden rows staged per pass of cluster_score_cc_kernel (32 KB)
constexpr int kHeadScoreTcRows = 16;   // more hidden rows than this: the scores on the tensor cores
constexpr int kHeadMaxVecs = 8;        // 16-byte vectors per lane of one embedding row: H <= 2048
constexpr int kHeadMaxClusters = 8192;  // cluster keys held in shared memory by cluster_topk_kernel
constexpr int kHeadMaxTopK = 256;
constexpr int kHeadMaxCand = 8192;     // candidates per row (sorted in shared memory)
constexpr int kHeadBitmapV = 262144;   // vocabularies up to this size are ranked through a bitmap

struct HeadParams {
  const __nv_bfloat16* hidden;     // [R, H]
  const __nv_bfloat16* centroids;  // [n_clusters, H]
  const __nv_bfloat16* W_ord;      // [V, H], cluster by cluster
  const int32_t* cluster_off;      // [n_clusters + 1]
  const int32_t* ord2tok;          // [V]
  float* scores;                   // [ksplit, R, n_clusters] partial scores (workspace)
  int32_t* sel;                    // [R, top_k] selected clusters (workspace)
  int32_t* pos;                    // [R, top_k + 1] candidate offsets (workspace)
  int32_t* out_tok;                // [R, max_cand]
  float* out_logit;                // [R, max_cand]
  int32_t* out_count;              // [R]
  int* status;
  int R, H, V, n_clusters, top_k, max_cand;
  int ksplit;                      // K parts of the score GEMM (partials to add)
};

// Dot product of one embedding row (held by the lanes: vector lane + 32k of
// the row, k < nv) with a bf16 row in shared memory, warp-reduced (lane 0's
// result is the one to use; every lane gets it).
__device__ __forceinline__ float dot_row_smem(const uint4 (&e)[kHeadMaxVecs], int nv, const uint4* hs) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < kHeadMaxVecs; ++k) {
    if (k < nv) {
      const uint4 a = e[k], b = hs[lane + 32 * k];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float a0, a1, b0, b1;
        bf16x2_unpack(aw[q], a0, a1);
        bf16x2_unpack(bw[q], b0, b1);
        acc = fmaf(a0, b0, acc);
        acc = fmaf(a1, b1, acc);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
}

__device__ __forceinline__ void load_row_vecs(const __nv_bfloat16* row, int nv, uint4 (&e)[kHeadMaxVecs]) {
  const int lane = threadIdx.x & 31;
  const uint4* v = reinterpret_cast<const uint4*>(row);
#pragma unroll
  for (int k = 0; k < kHeadMaxVecs; ++k)
    if (k < nv) e[k] = __ldg(v + lane + 32 * k);
}

// ---- 1a. cluster scores for few hidden rows, on the CUDA cores: grid
// ceil(n_clusters / kHeadWarps) x row blocks; each warp holds one centroid,
// the CTA stages kHeadRowBlock hidden rows in shared memory.  Up to 16 rows
// this measured faster than the tensor-core GEMM below (R = 4: 37.6 against
// 40.5 us per head call), whose split-K partials the selection must add ----
__global__ void __launch_bounds__(kHeadThreads, 1) cluster_score_cc_kernel(const __grid_constant__ HeadParams p) {
  __shared__ __align__(16) __nv_bfloat16 hs[kHeadRowBlock * kHeadMaxVecs * 32 * 8];
  grid_dep_launch();
  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = p.H / 256;  // 16-byte vectors per lane
  const int r0 = blockIdx.y * kHeadRowBlock;
  const int nr = min(kHeadRowBlock, p.R - r0);
  // stage the block's hidden rows
  const uint4* src = reinterpret_cast<const uint4*>(p.hidden + static_cast<size_t>(r0) * p.H);
  uint4* dst = reinterpret_cast<uint4*>(hs);
  for (int i = threadIdx.x; i < nr * (p.H / 8); i += kHeadThreads) {
    const int r = i / (p.H / 8), k = i - r * (p.H / 8);
    dst[r * kHeadMaxVecs * 32 + k] = __ldg(src + i);
  }
  __syncthreads();
  const int c = blockIdx.x * kHeadWarps + warp;
  if (c >= p.n_clusters) return;
  uint4 e[kHeadMaxVecs];
  load_row_vecs(p.centroids + static_cast<size_t>(c) * p.H, nv, e);
  for (int r = 0; r < nr; ++r) {
    const float z = dot_row_smem(e, nv, dst + r * kHeadMaxVecs * 32);
    if (lane == 0) p.scores[static_cast<size_t>(r0 + r) * p.n_clusters + c] = z;
  }
}

// ---- 1b. cluster scores on the tensor cores (more than 16 hidden rows) ----
// z[r, c] = h[r] . C[c] is a GEMM: A = 128 centroids (the MMA's M, the TMEM
// lanes), B = a chunk of N hidden rows (the MMA's N), K = H in stages of 64
// (128-byte swizzled rows) through a TMA ring.  Grid (tiles * ksplit, row
// chunks): CTA (tile, part) takes the K steps [part*kper, (part+1)*kper) and
// writes its partial sums to scores[part][r][c]; cluster_topk_kernel adds the
// parts in order.  Warp 0 lane 0 loads, warp 1 lane 0 issues the MMAs, then
// all four warps read the accumulator (warp w: TMEM lanes 32w..32w+31).
constexpr int kScThreads = 128;
constexpr int kScStages = 4;
constexpr int kScTileC = 128;                         // centroids per tile
constexpr int kScK = 64;                              // K per stage
constexpr int kScMaxN = 256;                          // hidden rows per CTA (MMA N)
constexpr int kScMaxSplit = 8;                        // K parts at most
constexpr uint32_t kScABytes = kScTileC * kScK * 2;  // 16 KB of centroids per stage

struct ScoreParams {
  CUtensorMap tmC;  // centroids [n_clusters, H] bf16, box 64 x 128
  CUtensorMap tmH;  // hidden [R, H] bf16, box 64 x N
  float* scores;    // [ksplit, R, n_clusters]
  int* status;
  int R, H, n_clusters, N, ksplit, kper;
};

__host__ __device__ inline uint32_t sc_stage_bytes(int N) { return kScABytes + static_cast<uint32_t>(N) * 128u; }
__host__ __device__ inline uint32_t sc_tmem_cols(int N) { return N <= 32 ? 32u : (N <= 64 ? 64u : (N <= 128 ? 128u : 256u)); }

__global__ void __launch_bounds__(kScThreads) cluster_score_tc_kernel(const __grid_constant__ ScoreParams p) {
  extern __shared__ __align__(1024) uint8_t sc_raw[];
  uint8_t* smem = sc_raw + ((1024u - (smem_u32(sc_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t full[kScStages], empty[kScStages], done;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / p.ksplit, part = blockIdx.x - tile * p.ksplit;
  const int ksteps = p.H / kScK;
  const int k0 = part * p.kper, nk = max(0, min(ksteps, k0 + p.kper) - k0);
  const uint32_t sbytes = sc_stage_bytes(p.N), ncols = sc_tmem_cols(p.N);
  grid_dep_launch();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kScStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_base, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  // the hidden rows may come from the previous kernel, and the previous call's
  // selection still reads the scores
  grid_dep_wait();
  if (warp == 0 && lane == 0) {
    int i = 0;
    for (; i < nk; ++i) {
      const int s = i % kScStages;
      if (i >= kScStages && !mbar_wait(&empty[s], ((i / kScStages) - 1) & 1, p.status, kWaitLimitCycles)) break;
      uint8_t* a = smem + s * sbytes;
      mbar_arrive_expect_tx(&full[s], sbytes);
      tma_load_2d(a, &p.tmC, (k0 + i) * kScK, tile * kScTileC, &full[s]);
      tma_load_2d(a + kScABytes, &p.tmH, (k0 + i) * kScK, static_cast<int>(blockIdx.y) * p.N, &full[s]);
    }
    // the copies of the last stages land before the CTA exits
    for (int j = (i > kScStages ? i - kScStages : 0); j < i; ++j)
      mbar_wait(&full[j % kScStages], (j / kScStages) & 1, p.status, kWaitLimitCycles);
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16_f32(kScTileC, p.N);
    bool ok = nk > 0;
    for (int i = 0; i < nk; ++i) {
      const int s = i % kScStages;
      if (!mbar_wait(&full[s], (i / kScStages) & 1, p.status, kWaitLimitCycles)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t ad = smem_desc_k128(smem_u32(smem + s * sbytes));
      const uint64_t bd = smem_desc_k128(smem_u32(smem + s * sbytes + kScABytes));
#pragma unroll
      for (int kk = 0; kk < kScK / 16; ++kk) tc_mma(tmem, ad + 2 * kk, bd + 2 * kk, idesc, i > 0 || kk > 0);
      tc_commit(&empty[s]);  // the stage is free once these MMAs have read it
    }
    if (ok)
      tc_commit(&done);
    else
      mbar_arrive(&done);  // status already set (or no K step): the epilogue stores nothing
  }
  __syncwarp();
  const bool got = mbar_wait(&done, 0, p.status, kWaitLimitCycles) && nk > 0;
  tc_fence_after();
  const int c = tile * kScTileC + warp * 32 + lane;
  const int r0 = static_cast<int>(blockIdx.y) * p.N;
  float* out = p.scores + static_cast<size_t>(part) * p.R * p.n_clusters;
  for (int g = 0; g < p.N; g += 32) {
    float v[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(g), v);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int r = r0 + g + j;
      if (got && g + j < p.N && r < p.R && c < p.n_clusters) out[static_cast<size_t>(r) * p.n_clusters + c] = v[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, ncols);
}

// Block-wide exclusive scan of one int per thread (all threads call); also
// returns the block total.  s_w: kHeadWarps ints of shared memory.
__device__ __forceinline__ int block_excl_scan(int v, int* s_w, int* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  int pre = 0, tot = 0;
  for (int w = 0; w < kHeadWarps; ++w) {
    const int x = s_w[w];
    if (w < warp) pre += x;
    tot += x;
  }
  __syncthreads();
  *total = tot;
  return pre + incl - v;
}

// ---- 2. top_k clusters of one row and their candidate offsets ----
// A radix select (tk_block_kth: 4 passes of 8-bit digits) finds the key of
// the top_k-th largest score; the clusters above it are kept, and of those
// equal to it the lowest indices.  Thread t owns the clusters
// [t*per, (t+1)*per), so the scans run in index order.  The selection is
// written in index order (its order does not matter: the candidates are
// sorted by token afterwards).
__global__ void __launch_bounds__(kHeadThreads, 1) cluster_topk_kernel(const __grid_constant__ HeadParams p) {
  extern __shared__ __align__(16) uint32_t keys[];  // [n_clusters]
  __shared__ int hist[256];
  __shared__ int s_w[kHeadWarps];
  __shared__ int s_val[2];
  grid_dep_launch();
  grid_dep_wait();
  const int r = blockIdx.x, t = threadIdx.x;
  const int Nc = p.n_clusters;
  // the K parts of the score GEMM, added in order; a thread's loads (four
  // clusters x every part) are all issued before the first add
  const float* z = p.scores + static_cast<size_t>(r) * Nc;
  const size_t part_stride = static_cast<size_t>(p.R) * Nc;
  constexpr int kCPer = 4;
  for (int c0 = t; c0 < Nc; c0 += kHeadThreads * kCPer) {
    float part[kCPer][kScMaxSplit];
#pragma unroll
    for (int i = 0; i < kCPer; ++i) {
      const int c = c0 + i * kHeadThreads;
#pragma unroll
      for (int q = 0; q < kScMaxSplit; ++q)
        part[i][q] = (c < Nc && q < p.ksplit) ? __ldcg(z + q * part_stride + c) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kCPer; ++i) {
      const int c = c0 + i * kHeadThreads;
      float zc = part[i][0];
#pragma unroll
      for (int q = 1; q < kScMaxSplit; ++q)
        if (q < p.ksplit) zc += part[i][q];
      if (c < Nc) keys[c] = logit_key(zc);
    }
  }
  __syncthreads();
  int greater;
  const uint32_t prefix = tk_block_kth(keys, Nc, p.top_k, hist, s_val, &greater);
  const int remaining = p.top_k - greater;  // keys equal to the k-th to take, lowest index first
  // prefix: the top_k-th largest key; keep keys above it and the `remaining`
  // lowest-index keys equal to it
  const int per = (Nc + kHeadThreads - 1) / kHeadThreads;
  const int c0 = min(Nc, t * per), c1 = min(Nc, c0 + per);
  int eq = 0;
  for (int c = c0; c < c1; ++c) eq += (keys[c] == prefix);
  int tot;
  int eq_before = block_excl_scan(eq, s_w, &tot);
  int nsel = 0;
  for (int c = c0; c < c1; ++c) {
    const uint32_t k = keys[c];
    nsel += (k > prefix) || (k == prefix && eq_before++ < remaining);
  }
  int sel_before = block_excl_scan(nsel, s_w, &tot);
  // sizes of the selected clusters, in the same order, for the candidate offsets
  int32_t* sel = p.sel + static_cast<size_t>(r) * p.top_k;
  int32_t* pos = p.pos + static_cast<size_t>(r) * (p.top_k + 1);
  eq_before = block_excl_scan(eq, s_w, &tot);
  int size_sum = 0;
  for (int c = c0; c < c1; ++c) {
    const uint32_t k = keys[c];
    if ((k > prefix) || (k == prefix && eq_before++ < remaining))
      size_sum += max(0, min(p.cluster_off[c + 1], p.V) - max(p.cluster_off[c], 0));
  }
  int total;
  int size_before = block_excl_scan(size_sum, s_w, &total);
  eq_before = block_excl_scan(eq, s_w, &tot);
  for (int c = c0; c < c1; ++c) {
    const uint32_t k = keys[c];
    if ((k > prefix) || (k == prefix && eq_before++ < remaining)) {
      if (sel_before < p.top_k) {
        sel[sel_before] = c;
        pos[sel_before] = size_before;
      }
      ++sel_before;
      size_before += max(0, min(p.cluster_off[c + 1], p.V) - max(p.cluster_off[c], 0));
    }
  }
  if (t == 0) {
    pos[p.top_k] = total;
    if (total > p.max_cand) atomicOr(p.status, kStatusLimit);
    p.out_count[r] = min(total, p.max_cand);
  }
}

// ---- 3. candidate logits: grid (top_k, R), one warp per token row ----
__global__ void __launch_bounds__(kHeadThreads, 1) cand_logit_kernel(const __grid_constant__ HeadParams p) {
  __shared__ __align__(16) __nv_bfloat16 hs[kHeadMaxVecs * 32 * 8];
  grid_dep_launch();
  const int k = blockIdx.x, r = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = p.H / 256;
  // the hidden row is an input: staged before waiting for the selection
  const uint4* src = reinterpret_cast<const uint4*>(p.hidden + static_cast<size_t>(r) * p.H);
  for (int i = threadIdx.x; i < p.H / 8; i += kHeadThreads) reinterpret_cast<uint4*>(hs)[i] = __ldg(src + i);
  grid_dep_wait();
  __syncthreads();
  const int c = p.sel[static_cast<size_t>(r) * p.top_k + k];
  if (c < 0 || c >= p.n_clusters) return;  // see cluster_topk_kernel
  const int base = p.pos[static_cast<size_t>(r) * (p.top_k + 1) + k];
  const int i0 = max(p.cluster_off[c], 0), i1 = min(p.cluster_off[c + 1], p.V);
  int32_t* otok = p.out_tok + static_cast<size_t>(r) * p.max_cand;
  float* olog = p.out_logit + static_cast<size_t>(r) * p.max_cand;
  // two embedding rows in flight per warp
  for (int i = i0 + 2 * warp; i < i1; i += 2 * kHeadWarps) {
    const int slot = base + (i - i0);
    if (slot >= p.max_cand) break;  // overflow: reported by the selection kernel
    const bool two = (i + 1 < i1) && (slot + 1 < p.max_cand);
    uint4 e0[kHeadMaxVecs], e1[kHeadMaxVecs];
    load_row_vecs(p.W_ord + static_cast<size_t>(i) * p.H, nv, e0);
    if (two) load_row_vecs(p.W_ord + static_cast<size_t>(i + 1) * p.H, nv, e1);
    const float l0 = dot_row_smem(e0, nv, reinterpret_cast<const uint4*>(hs));
    const float l1 = two ? dot_row_smem(e1, nv, reinterpret_cast<const uint4*>(hs)) : 0.f;
    if (lane == 0) {
      otok[slot] = p.ord2tok[i];
      olog[slot] = l0;
      if (two) {
        otok[slot + 1] = p.ord2tok[i + 1];
        olog[slot + 1] = l1;
      }
    }
  }
}

// ---- 4. sort one row's candidates by token id (ascending) ----
// Tokens are distinct ids in [0, V): for V <= kHeadBitmapV a candidate's rank
// is the number of candidate tokens below it, read off a V-bit bitmap with a
// prefix of its words' population counts (no comparison sort).  Larger
// vocabularies use a bitonic sort of (token, logit) keys.
constexpr size_t kHeadSortSmemBitmap = static_cast<size_t>(kHeadMaxCand) * 8 + (kHeadBitmapV / 32) * 8;

__global__ void __launch_bounds__(kHeadThreads, 1) cand_sort_kernel(const __grid_constant__ HeadParams p) {
  extern __shared__ __align__(16) unsigned long long dyn[];
  __shared__ int s_w[kHeadWarps];
  grid_dep_launch();
  grid_dep_wait();
  const int r = blockIdx.x, t = threadIdx.x;
  const int n = p.out_count[r];
  int32_t* otok = p.out_tok + static_cast<size_t>(r) * p.max_cand;
  float* olog = p.out_logit + static_cast<size_t>(r) * p.max_cand;
  if (p.V <= kHeadBitmapV) {
    int32_t* st_tok = reinterpret_cast<int32_t*>(dyn);
    float* st_log = reinterpret_cast<float*>(st_tok + kHeadMaxCand);
    uint32_t* bits = reinterpret_cast<uint32_t*>(st_log + kHeadMaxCand);
    int* wpre = reinterpret_cast<int*>(bits + kHeadBitmapV / 32);
    const int nw = (p.V + 31) / 32;
    for (int i = t; i < nw; i += kHeadThreads) bits[i] = 0u;
    // the candidates into shared memory, all of a thread's loads issued
    // before its stores (n <= kHeadMaxCand = 16 per thread)
    {
      constexpr int kPer = kHeadMaxCand / kHeadThreads;
      int32_t tk[kPer];
      float lg[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = t + j * kHeadThreads;
        tk[j] = (i < n) ? __ldcg(otok + i) : 0;
        lg[j] = (i < n) ? __ldcg(olog + i) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = t + j * kHeadThreads;
        if (i < n) {
          st_tok[i] = tk[j];
          st_log[i] = lg[j];
        }
      }
    }
    __syncthreads();
    for (int i = t; i < n; i += kHeadThreads) {
      const int x = st_tok[i];
      if (x >= 0 && x < p.V) atomicOr(&bits[x >> 5], 1u << (x & 31));
    }
    __syncthreads();
    const int per = (nw + kHeadThreads - 1) / kHeadThreads;
    const int w0 = min(nw, t * per), w1 = min(nw, w0 + per);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
    int tot;
    int run = block_excl_scan(cnt, s_w, &tot);
    for (int w = w0; w < w1; ++w) {
      wpre[w] = run;
      run += __popc(bits[w]);
    }
    __syncthreads();
    for (int i = t; i < n; i += kHeadThreads) {
      const int x = st_tok[i];
      if (x < 0 || x >= p.V) continue;  // not a token id: dropped
      const int rank = wpre[x >> 5] + __popc(bits[x >> 5] & ((1u << (x & 31)) - 1u));
      if (rank < n) {
        otok[rank] = x;
        olog[rank] = st_log[i];
      }
    }
    return;
  }
  unsigned long long* sk = dyn;
  const int n2 = tk_pow2(max(n, 1));
  // key: complemented token (descending sort = ascending tokens), then the
  // logit's bits; padding keys are 0 and sort last
  for (int i = t; i < n2; i += kHeadThreads)
    sk[i] = (i < n) ? (static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(otok[i])) << 32) |
                          __float_as_uint(olog[i])
                    : 0ull;
  __syncthreads();
  tk_sort_desc(sk, n2);
  for (int i = t; i < n; i += kHeadThreads) {
    otok[i] = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(sk[i] >> 32));
    olog[i] = __uint_as_float(static_cast<uint32_t>(sk[i] & 0xffffffffull));
  }
}

}  // namespace specv
