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
//   cluster_score_kernel   z[r, c] = h[r] . C[c]  (fp32 sums of bf16 products;
//                          each warp holds one centroid, the CTA stages
//                          kHeadRowBlock hidden rows in shared memory)
//   cluster_topk_kernel    one CTA per row: bitonic sort of (score, -index)
//                          keys; the top_k clusters (the lowest index first
//                          among equal scores) and their candidate offsets
//   cand_logit_kernel      grid (top_k, R): one CTA per selected cluster, one
//                          warp per token row, writes (token, logit) unsorted
//   cand_sort_kernel       one CTA per row: sorts the candidates by token id
//                          (the order the sparse verification searches in)
// The bulk of the bytes is the gathered embedding rows (top_k clusters of
// about V / n_clusters rows of 2H bytes per hidden row): HBM/L2 bound.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "topkp.cuh"

namespace specv {

constexpr int kHeadThreads = 512;  // tk_sort_desc assumes 512-thread CTAs
constexpr int kHeadWarps = kHeadThreads / 32;
constexpr int kHeadRowBlock = 4;       // hidden rows staged per pass of cluster_score_kernel (32 KB)
constexpr int kHeadMaxVecs = 16;       // 16-byte vectors per lane of one embedding row: H <= 4096
constexpr int kHeadMaxClusters = 8192;  // sorted in shared memory by cluster_topk_kernel
constexpr int kHeadMaxTopK = 256;
constexpr int kHeadMaxCand = 8192;     // candidates per row (sorted in shared memory)

struct HeadParams {
  const __nv_bfloat16* hidden;     // [R, H]
  const __nv_bfloat16* centroids;  // [n_clusters, H]
  const __nv_bfloat16* W_ord;      // [V, H], cluster by cluster
  const int32_t* cluster_off;      // [n_clusters + 1]
  const int32_t* ord2tok;          // [V]
  float* scores;                   // [R, n_clusters] (workspace)
  int32_t* sel;                    // [R, top_k] selected clusters (workspace)
  int32_t* pos;                    // [R, top_k + 1] candidate offsets (workspace)
  int32_t* out_tok;                // [R, max_cand]
  float* out_logit;                // [R, max_cand]
  int32_t* out_count;              // [R]
  int* status;
  int R, H, V, n_clusters, top_k, max_cand;
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

// ---- 1. cluster scores: grid ceil(n_clusters / kHeadWarps) x row blocks ----
__global__ void __launch_bounds__(kHeadThreads, 1) cluster_score_kernel(const __grid_constant__ HeadParams p) {
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

// ---- 2. top_k clusters of one row and their candidate offsets ----
__global__ void __launch_bounds__(kHeadThreads, 1) cluster_topk_kernel(const __grid_constant__ HeadParams p) {
  extern __shared__ __align__(16) unsigned long long sk[];  // [n2] keys
  grid_dep_launch();
  grid_dep_wait();
  const int r = blockIdx.x;
  const int n2 = tk_pow2(p.n_clusters);
  const float* z = p.scores + static_cast<size_t>(r) * p.n_clusters;
  // key: the score's order-preserving bits, then the complemented index, so
  // that a descending sort puts the lowest index first among equal scores
  for (int c = threadIdx.x; c < n2; c += kHeadThreads)
    sk[c] = (c < p.n_clusters)
                ? (static_cast<unsigned long long>(logit_key(z[c])) << 32) | (0xffffffffu - static_cast<uint32_t>(c))
                : 0ull;
  __syncthreads();
  tk_sort_desc(sk, n2);
  int32_t* sel = p.sel + static_cast<size_t>(r) * p.top_k;
  for (int k = threadIdx.x; k < p.top_k; k += kHeadThreads)
    sel[k] = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(sk[k] & 0xffffffffull));
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t* pos = p.pos + static_cast<size_t>(r) * (p.top_k + 1);
    int total = 0;
    for (int k = 0; k < p.top_k; ++k) {
      const int c = static_cast<int>(0xffffffffu - static_cast<uint32_t>(sk[k] & 0xffffffffull));
      pos[k] = total;
      // a padding key (possible only with NaN scores) decodes to c >= n_clusters: an empty cluster
      if (c < p.n_clusters) total += max(0, min(p.cluster_off[c + 1], p.V) - max(p.cluster_off[c], 0));
    }
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
  for (int i = i0 + warp; i < i1; i += kHeadWarps) {
    const int slot = base + (i - i0);
    if (slot >= p.max_cand) break;  // overflow: reported by the selection kernel
    uint4 e[kHeadMaxVecs];
    load_row_vecs(p.W_ord + static_cast<size_t>(i) * p.H, nv, e);
    const float lg = dot_row_smem(e, nv, reinterpret_cast<const uint4*>(hs));
    if (lane == 0) {
      otok[slot] = p.ord2tok[i];
      olog[slot] = lg;
    }
  }
}

// ---- 4. sort one row's candidates by token id (ascending) ----
__global__ void __launch_bounds__(kHeadThreads, 1) cand_sort_kernel(const __grid_constant__ HeadParams p) {
  extern __shared__ __align__(16) unsigned long long sk[];
  grid_dep_launch();
  grid_dep_wait();
  const int r = blockIdx.x;
  const int n = p.out_count[r];
  const int n2 = tk_pow2(max(n, 1));
  int32_t* otok = p.out_tok + static_cast<size_t>(r) * p.max_cand;
  float* olog = p.out_logit + static_cast<size_t>(r) * p.max_cand;
  // key: complemented token (descending sort = ascending tokens), then the
  // logit's bits; padding keys are 0 and sort last
  for (int i = threadIdx.x; i < n2; i += kHeadThreads)
    sk[i] = (i < n) ? (static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(otok[i])) << 32) |
                          __float_as_uint(olog[i])
                    : 0ull;
  __syncthreads();
  tk_sort_desc(sk, n2);
  for (int i = threadIdx.x; i < n; i += kHeadThreads) {
    otok[i] = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(sk[i] >> 32));
    olog[i] = __uint_as_float(static_cast<uint32_t>(sk[i] & 0xffffffffull));
  }
}

}  // namespace specv
