// topkp.cuh — verification with top-k / top-p truncation applied identically
// to the target and the draft distributions ("Gemma 4 Multi-Token Prediction
// (MTP) 深度解析" §5.1 samples with top_k=64, top_p=0.95 next to the drafter;
// "第 8 章 投机解码：一次前向，验证好几个字", 为什么输出不会变: whatever transforms
// the target distribution must transform the draft distribution the same way).
//
// Per row (temperature T, ks = log2(e)/T):
//   K  = entries with fewer than top_k strictly larger logits (ties stay);
//   pk = softmax over K;
//   K' = entries of K whose strictly more likely entries hold less than top_p
//        of pk (tie groups stay together; the most likely entries always stay);
//   p' = softmax over K', 0 elsewhere.
//
//   topk_select_kernel  one CTA per row: a superset of K from the row
//                       reducer's block maxima (the blocks whose maximum
//                       reaches the top_k-th largest block maximum), else a
//                       radix select of the top_k-th largest logit over
//                       order-preserving keys; a sort by (logit desc, index
//                       asc), the top-p cut from a two-float prefix scan, and
//                       the kept list re-sorted by vocabulary index.
//   topkp_tail_kernel   one CTA per sequence: the decision on p'(d)/q'(d)
//                       (binary search in the kept lists), then the draw by
//                       inverse CDF over the kept list of row n (residual
//                       max(0, p'_n - q'_n), nonzero only where p'_n is) or of
//                       row gamma (bonus), in ascending vocabulary order.
#pragma once

#include <cfloat>
#include <climits>
#include <cuda_bf16.h>

#include "common.cuh"
#include "decide.cuh"
#include "sample.cuh"

namespace specv {

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkMaxK = 1024;   // top_k limit
constexpr int kTkStore = 2048;  // kept entries per row, ties included (beyond: status error)

struct TopkParams {
  const void* target;        // [B, gamma+1, V]
  const void* draft;         // [B, gamma, V]
  const float* temperature;  // [B]
  int* list_idx;             // [B*(2*gamma+1)][kTkStore] kept entries, ascending vocabulary index
  float* list_val;           // same layout: their raw logits
  float4* rowtk;             // [B*(2*gamma+1)] {count bits, mk, log2 S', argmax bits}
  float2* rowd;              // [B*(2*gamma+1)] {logit of the row's draft token, 1 if kept else 0}
  const int32_t* draft_tokens;  // [B, gamma]
  int* status;
  // the maxima of the row reducer's 32-vector blocks, from which the select
  // kernel bounds K (nullptr: it finds K on its own)
  const float* submax;  // [B*(2*gamma+1)*cpr*kVecPerLane]
  int B, gamma, V, top_k, cpr, CE;
  float top_p;
};

// Order-preserving key of a logit: larger value <=> larger unsigned key
// (-0 is folded onto +0 so that equal values have equal keys).
__device__ __forceinline__ uint32_t logit_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// Vectors of a row visited by a pass: all of them, or the sample -- the
// first 16 entries of every 256 (contiguous, so the sample costs 1/16 of the
// row's sectors).
template <typename T>
struct TkRange {
  static constexpr int P = Elt<T>::kPerVec;
  static constexpr int kVpb = 256 / P, kSpb = 16 / P;  // vectors per block of 256, sampled per block
  int nvec;
  bool sample;
  __device__ __forceinline__ int count() const {
    return sample ? (nvec / kVpb) * kSpb + min(kSpb, nvec % kVpb) : nvec;
  }
  __device__ __forceinline__ int vec(int i) const { return sample ? (i / kSpb) * kVpb + (i % kSpb) : i; }
};

// One pass of the radix select: counts, per 8-bit digit at `shift`, the
// visited entries whose key agrees with `prefix` on the bits above it.
template <typename T>
__device__ __forceinline__ void tk_histogram(const void* row, const TkRange<T>& rg, uint32_t prefix, uint32_t pmask,
                                             int shift, int* hist /* [kTkWarps][256] */) {
  constexpr int P = Elt<T>::kPerVec;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kBatch = 4;  // vectors in flight per thread
  const uint4* v4 = reinterpret_cast<const uint4*>(row);
  const int n = rg.count();
  int* h = hist + warp * 256;
  for (int base = 0; base < n; base += kBatch * kTkThreads) {  // block-uniform
    uint4 u[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = base + j * kTkThreads + threadIdx.x;
      u[j] = (i < n) ? __ldg(v4 + rg.vec(i)) : neg_inf_vec<T>();
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = base + j * kTkThreads + threadIdx.x;
      float x[P];
      Elt<T>::unpack(u[j], x);
#pragma unroll
      for (int k = 0; k < P; ++k) {
        const uint32_t key = logit_key(x[k]);
        const bool in = (i < n) && ((key & pmask) == prefix);
        const int digit = in ? static_cast<int>((key >> shift) & 255u) : 256;
        const unsigned same = __match_any_sync(0xffffffffu, digit);
        if (in && lane == __ffs(same) - 1) atomicAdd(&h[digit], __popc(same));
      }
    }
  }
}

// Radix select over the visited entries: the significant key bits (prefix,
// pmask) of the rank-th largest.  Block-wide; hist is [kTkWarps][256].
template <typename T>
__device__ __noinline__ void tk_radix_select(const void* row, const TkRange<T>& rg, int rank, int* hist,
                                             int* s_digit, int* s_remaining, uint32_t* prefix_out,
                                             uint32_t* pmask_out) {
  constexpr int kPasses = (sizeof(T) == 2) ? 2 : 4;  // bf16 keys carry 16 significant bits
  uint32_t prefix = 0, pmask = 0;
  if (threadIdx.x == 0) *s_remaining = rank;
#pragma unroll 1
  for (int pass = 0; pass < kPasses; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < kTkWarps * 256; i += kTkThreads) hist[i] = 0;
    __syncthreads();
    tk_histogram<T>(row, rg, prefix, pmask, shift, hist);
    __syncthreads();
    if (threadIdx.x < 256) {
      int tot = 0;
      for (int w = 0; w < kTkWarps; ++w) tot += hist[w * 256 + threadIdx.x];
      hist[threadIdx.x] = tot;  // row 0 now holds the totals (each thread touches only its digit)
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // the digit holding the rank-th largest: lane l owns digits 255-8l ..
      // 248-8l (descending), a warp scan gives the counts above each lane
      const int lane = threadIdx.x, rem = *s_remaining;
      int c[8], own = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        c[q] = hist[255 - 8 * lane - q];
        own += c[q];
      }
      int incl = own;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const int above = incl - own;  // entries in the digits above this lane's
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= rem && above < rem);
      if (lane == __ffs(hit) - 1) {
        int cum = above, d = 255 - 8 * lane;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (cum + c[q] >= rem) {
            d = 255 - 8 * lane - q;
            break;
          }
          cum += c[q];
        }
        *s_digit = d;
        *s_remaining = rem - cum;
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(*s_digit) << shift;
    pmask |= 255u << shift;
    __syncthreads();
  }
  *prefix_out = prefix;
  *pmask_out = pmask;
}

// Every entry of the row whose significant key bits reach (prefix, pmask),
// packed (key, ~index) into sk (at most kTkStore kept); returns the count of
// all such entries.  Each thread marks the hits of its batch of vectors in a
// bit mask (a vector is looked at element by element only when its maximum
// reaches the threshold); one warp scan and one shared-memory atomic per
// batch place them.
template <typename T>
__device__ __noinline__ int tk_collect(const void* row, int V, uint32_t prefix, uint32_t pmask,
                                       unsigned long long* sk, int* s_count) {
  constexpr int P = Elt<T>::kPerVec;
  constexpr int kBatch = 8;  // vectors in flight per thread
  static_assert(kBatch * P <= 64, "hit mask");
  const int lane = threadIdx.x & 31;
  const uint4* v4 = reinterpret_cast<const uint4*>(row);
  const int nvec = V / P;
  if (threadIdx.x == 0) *s_count = 0;
  __syncthreads();
  for (int base = 0; base < nvec; base += kBatch * kTkThreads) {  // block-uniform
    uint4 u[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = base + j * kTkThreads + threadIdx.x;
      u[j] = (i < nvec) ? __ldg(v4 + i) : neg_inf_vec<T>();
    }
    unsigned long long hits = 0ull;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const bool inb = base + j * kTkThreads + static_cast<int>(threadIdx.x) < nvec;
      if (inb && (logit_key(vec_max<T>(u[j])) & pmask) >= prefix) {
        float x[P];
        Elt<T>::unpack(u[j], x);
#pragma unroll
        for (int e = 0; e < P; ++e)
          if ((logit_key(x[e]) & pmask) >= prefix) hits |= 1ull << (j * P + e);
      }
    }
    const int nh = __popcll(hits);
    int inc = nh;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += o;
    }
    const int total = __shfl_sync(0xffffffffu, inc, 31);
    if (total == 0) continue;  // warp-uniform
    int pos = 0;
    if (lane == 31) pos = atomicAdd(s_count, total);
    pos = __shfl_sync(0xffffffffu, pos, 31) + inc - nh;
    while (hits) {
      const int bit = __ffsll(static_cast<long long>(hits)) - 1;
      hits &= hits - 1ull;
      const int j = bit / P, e = bit - j * P;
      if (pos < kTkStore) {
        uint4 uj = u[0];
#pragma unroll
        for (int jj = 1; jj < kBatch; ++jj) uj = (jj == j) ? u[jj] : uj;
        float x[P];
        Elt<T>::unpack(uj, x);
        float xe = x[0];
#pragma unroll
        for (int ee = 1; ee < P; ++ee) xe = (ee == e) ? x[ee] : xe;
        const uint32_t idx = static_cast<uint32_t>((base + j * kTkThreads + threadIdx.x) * P + e);
        sk[pos] = (static_cast<unsigned long long>(logit_key(xe)) << 32) | (0xffffffffu - idx);
      }
      ++pos;
    }
  }
  __syncthreads();
  return *s_count;
}

// Block-wide bitonic sort of n_pow2 (<= 2048) 64-bit keys in shared memory,
// descending.  Pair i of a stage is handled by thread i mod kTkThreads.  For a
// stride of at most 32 the pairs of a warp lie in that warp's own 64-entry
// blocks (the same blocks at every such stride), so between two such stages a
// warp barrier suffices; any stage with a wider stride is fenced by block
// barriers.
__device__ __forceinline__ void tk_sort_desc(unsigned long long* a, int n_pow2) {
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n_pow2 / 2; i += kTkThreads) {
        // (i / stride) * 2 * stride + i % stride, stride a power of two
        const int lo = ((i & ~(stride - 1)) << 1) | (i & (stride - 1)), hi = lo + stride;
        const bool desc = ((lo & size) == 0);
        const unsigned long long x = a[lo], y = a[hi];
        if ((x < y) == desc) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      const int next = (stride > 1) ? (stride >> 1) : size;  // the next stage's stride
      const bool last = (stride == 1 && size == n_pow2);
      if (last || stride > 32 || next > 32) __syncthreads();
      else __syncwarp();
    }
  }
}

// Block-wide inclusive scan of one two-float value per thread (all threads
// call); also returns the block total.
__device__ __forceinline__ F2 tk_block_scan(F2 v, F2* s_wtot, F2* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  F2 incl = warp_scan_incl(v);
  if (lane == 31) s_wtot[warp] = incl;
  __syncthreads();
  F2 pre = f2_from(0.f), tot = f2_from(0.f);
  for (int w = 0; w < kTkWarps; ++w) {
    if (w < warp) pre = f2_add(pre, s_wtot[w]);
    tot = f2_add(tot, s_wtot[w]);
  }
  __syncthreads();
  *total = tot;
  return f2_add(incl, pre);
}

// Next power of two >= n (n >= 1).
__device__ __forceinline__ int tk_pow2(int n) {
  int p2 = 1;
  while (p2 < n) p2 <<= 1;
  return p2;
}

// Block-wide radix select over n keys in shared memory (`passes` passes of
// 8-bit digits, most significant first): the k-th largest key (1 <= k <= n),
// or, with fewer than 4 passes, its leading 8*passes bits (the rest zero) --
// exact as a threshold when the keys carry no more significant bits than
// that, as the keys of bf16 values carry 16.  *greater receives how many keys
// are strictly larger.  All threads call; every thread returns the same.
__device__ __forceinline__ uint32_t tk_block_kth(const uint32_t* keys, int n, int k, int* hist, int* s_val,
                                                 int* greater, int passes = 4) {
  const int t = threadIdx.x;
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = t; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int c = t; c < n; c += blockDim.x) {
      const uint32_t key = keys[c];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (t < 32) {
      // lane l owns digits 255-8l .. 248-8l; the digit reached by `remaining`
      int cnt[8], mine = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        cnt[q] = hist[255 - 8 * t - q];
        mine += cnt[q];
      }
      int incl = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (t >= off) incl += o;
      }
      int run = incl - mine;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (run < remaining && run + cnt[q] >= remaining) {
          s_val[0] = 255 - 8 * t - q;
          s_val[1] = run;
        }
        run += cnt[q];
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(s_val[0]) << shift;
    mask |= 255u << shift;
    remaining -= s_val[1];
    __syncthreads();
  }
  *greater = k - remaining;
  return prefix;
}

constexpr int kTkCollectMaxBlocks = 4096;  // block maxima held in shared memory
constexpr int kTkGatherBatch = 8;          // qualifying blocks in flight per warp
constexpr int kTkRankSortMax = 256;        // longer lists take the bitonic sort

// A superset of K from the row reducer's block maxima.  Those maxima are
// logits of the row, so the k-th largest of them, M_k, is a lower bound on the
// k-th largest logit: K lies inside the blocks whose maximum reaches M_k.  The
// qualifying blocks are compacted in order, the warps gather them
// kTkGatherBatch at a time (one 16-byte vector per lane) and append every
// logit >= M_k to sk as (key << 32 | ~index).  Returns how many there are
// (sk holds the first kTkStore).  `ck` is scratch for kTkCollectMaxBlocks keys
// and qlist for as many block numbers.
template <typename T>
__device__ __noinline__ int tk_gather_blocks(const TopkParams& p, int slot, const void* row, int k,
                                             uint32_t* ck, uint16_t* qlist, int* hist256, int* s_val, int* s_w,
                                             unsigned long long* sk, int* s_count) {
  constexpr int P = Elt<T>::kPerVec;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = p.cpr * kVecPerLane;
  const float* sm = p.submax + static_cast<size_t>(slot) * nb;
  for (int c = threadIdx.x; c < nb; c += kTkThreads) ck[c] = logit_key(__ldcg(sm + c));
  if (threadIdx.x == 0) *s_count = 0;
  __syncthreads();
  int greater;  // unused: the list keeps every logit >= the bound
  const uint32_t thr = tk_block_kth(ck, nb, k, hist256, s_val, &greater, sizeof(T) == 2 ? 2 : 4);  // k < nb
  // the qualifying blocks, compacted in order: thread t checks blocks
  // [t*per, (t+1)*per), a block scan gives each its position
  const int per = (nb + kTkThreads - 1) / kTkThreads;
  const int q0 = min(nb, static_cast<int>(threadIdx.x) * per), q1 = min(nb, q0 + per);
  int mine = 0;
  for (int q = q0; q < q1; ++q) mine += (ck[q] >= thr);
  int incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  int before = incl - mine, nq = 0;
  for (int w = 0; w < kTkWarps; ++w) {
    if (w < warp) before += s_w[w];
    nq += s_w[w];
  }
  for (int q = q0; q < q1; ++q)
    if (ck[q] >= thr) qlist[before++] = static_cast<uint16_t>(q);
  __syncthreads();
  // block q of chunk c covers the row's vectors c*CE/P + 32j .. +31 (q = 8c + j)
  const uint4* v4 = static_cast<const uint4*>(row);
  const int nvec_row = p.V / P, vpc = p.CE / P;
  for (int qb = warp; qb < nq; qb += kTkWarps * kTkGatherBatch) {  // warp-uniform
    // the batch's loads first (the only registers they hold are the data);
    // this lane's vector of block q = 8c + j is c*CE/P + 32j + lane
    uint4 u[kTkGatherBatch];
#pragma unroll
    for (int j = 0; j < kTkGatherBatch; ++j) {
      const int qi = qb + j * kTkWarps;
      const int q = (qi < nq) ? qlist[qi] : 0;
      const int c = q / kVecPerLane, jb = q - c * kVecPerLane;
      const int vi = c * vpc + 32 * jb + lane;
      const bool in = qi < nq && (32 * jb + lane) < vpc && vi < nvec_row;
      u[j] = in ? __ldg(v4 + vi) : neg_inf_vec<T>();
    }
#pragma unroll
    for (int j = 0; j < kTkGatherBatch; ++j) {
      const int qi = qb + j * kTkWarps;
      if (qi >= nq) break;  // warp-uniform
      const int q = qlist[qi];
      const int c = q / kVecPerLane, jb = q - c * kVecPerLane;
      const int vi = c * vpc + 32 * jb + lane;
      const bool in = (32 * jb + lane) < vpc && vi < nvec_row;
      float x[P];
      Elt<T>::unpack(u[j], x);
      uint32_t hits = 0;
#pragma unroll
      for (int e = 0; e < P; ++e)
        if (in && logit_key(x[e]) >= thr) hits |= 1u << e;
      const int nh = __popc(hits);
      int inc = nh;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
      }
      const int total = __shfl_sync(0xffffffffu, inc, 31);
      if (total == 0) continue;  // warp-uniform
      int base = 0;
      if (lane == 31) base = atomicAdd(s_count, total);
      base = __shfl_sync(0xffffffffu, base, 31) + inc - nh;
#pragma unroll
      for (int e = 0; e < P; ++e) {
        if ((hits >> e) & 1u) {
          if (base < kTkStore) {
            const uint32_t idx = static_cast<uint32_t>(vi * P + e);
            sk[base] = (static_cast<unsigned long long>(logit_key(x[e])) << 32) | (0xffffffffu - idx);
          }
          ++base;
        }
      }
    }
  }
  __syncthreads();
  return *s_count;
}

// Sort of n distinct 64-bit keys in shared memory, descending.  Up to
// kTkRankSortMax keys: each key goes to its rank (the number of larger keys)
// in tmp and back, one pass.  Longer lists: padded with zeros to a power of
// two and sorted by tk_sort_desc (the zeros end up behind the n keys).
__device__ __forceinline__ void tk_sort_keys_desc(unsigned long long* a, int n, unsigned long long* tmp) {
  if (n <= kTkRankSortMax) {
    for (int i = threadIdx.x; i < n; i += kTkThreads) {
      const unsigned long long x = a[i];
      int r = 0;
#pragma unroll 4
      for (int j = 0; j < n; ++j) r += (a[j] > x) ? 1 : 0;
      tmp[r] = x;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kTkThreads) a[i] = tmp[i];
    __syncthreads();
    return;
  }
  const int n2 = tk_pow2(n);
  for (int i = n + threadIdx.x; i < n2; i += kTkThreads) a[i] = 0ull;
  __syncthreads();
  tk_sort_desc(a, n2);
  __syncthreads();
}

constexpr int kTkWarpList = 128;  // lists finished by one warp (4 entries per lane)

__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Rank sort of n <= kTkWarpList distinct keys by one warp, descending.
__device__ __forceinline__ void tk_warp_sort_desc(unsigned long long* a, int n, unsigned long long* tmp) {
  const int lane = threadIdx.x & 31;
  for (int i = lane; i < n; i += 32) {
    const unsigned long long x = a[i];
    int r = 0;
#pragma unroll 4
    for (int j = 0; j < n; ++j) r += (a[j] > x) ? 1 : 0;
    tmp[r] = x;
  }
  __syncwarp();
  for (int i = lane; i < n; i += 32) a[i] = tmp[i];
  __syncwarp();
}

// The select kernel's work after K's superset is in sk, for a list of at
// most kTkWarpList entries, by one warp: the same steps and the same
// arithmetic as the block-wide path (whose scans reduce to warp 0's when
// every entry sits in warp 0), without block barriers.
__device__ __noinline__ void tk_finish_warp(const TopkParams& p, int slot, int k, int count, bool greedy,
                                            float temp, int dtok, unsigned long long* sk,
                                            unsigned long long* tmp) {
  const int lane = threadIdx.x & 31;
  tk_warp_sort_desc(sk, count, tmp);  // logit descending, index ascending
  {
    // K: the entries whose key reaches the k-th largest; ties with it stay
    const uint32_t kth = static_cast<uint32_t>(sk[min(k, count) - 1] >> 32);
    int c = count;
    for (int j = k + lane; j < count; j += 32)
      if (static_cast<uint32_t>(sk[j] >> 32) < kth) c = min(c, j);
    count = warp_min_i(c);
  }
  const int argmax = static_cast<int>(0xffffffffu - static_cast<uint32_t>(sk[0] & 0xffffffffull));
  if (greedy) {
    if (lane == 0) p.rowtk[slot] = make_float4(__int_as_float(0), kNegHuge, 0.f, __int_as_float(argmax));
    return;
  }
  // ---- softmax over K, the top-p cut, the normaliser of K' ----
  const float ks = kLog2e / temp;
  const float mk = key_logit(static_cast<uint32_t>(sk[0] >> 32)) * ks;
  float e[4];
  uint32_t kj[4];
  F2 my = f2_from(0.f);
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // this lane's entries 4l .. 4l+3
    const int j = 4 * lane + q;
    kj[q] = (j < count) ? static_cast<uint32_t>(sk[j] >> 32) : 0u;
    e[q] = (j < count) ? ex2(fmaf(key_logit(kj[q]), ks, -mk)) : 0.f;
    my = f2_add(my, f2_from(e[q]));
  }
  const int jprev = 4 * lane - 1;
  const uint32_t kprev = (jprev >= 0 && jprev < count) ? static_cast<uint32_t>(sk[jprev] >> 32) : 0xffffffffu;
  const F2 incl = warp_scan_incl(my);
  const F2 S = {__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
  int cut = count;
  if (p.top_p < 1.f) {
    const F2 thr = f2_mul_f(S, p.top_p);
    F2 run = f2_sub(incl, my);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = 4 * lane + q;
      if (j < count) {
        const bool start = (j == 0) || (kj[q] != (q == 0 ? kprev : kj[q - 1]));
        if (start && !f2_gt(thr, run)) cut = min(cut, j);
        run = f2_add(run, f2_from(e[q]));
      }
    }
    cut = warp_min_i(cut);
  }
  F2 my2 = f2_from(0.f);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (4 * lane + q < cut) my2 = f2_add(my2, f2_from(e[q]));
  const F2 incl2 = warp_scan_incl(my2);
  const float lse2 = log2f(__shfl_sync(0xffffffffu, incl2.hi, 31) + __shfl_sync(0xffffffffu, incl2.lo, 31));
  // ---- K' re-sorted by vocabulary index, written out ----
  unsigned long long mine[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = 4 * lane + q;
    mine[q] = 0ull;
    if (j < cut) {
      const uint32_t idx = 0xffffffffu - static_cast<uint32_t>(sk[j] & 0xffffffffull);
      mine[q] = (static_cast<unsigned long long>(0xffffffffu - idx) << 32) | kj[q];
    }
  }
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (4 * lane + q < cut) sk[4 * lane + q] = mine[q];
  __syncwarp();
  tk_warp_sort_desc(sk, cut, tmp);  // index ascending
  int* li = p.list_idx + static_cast<size_t>(slot) * kTkStore;
  float* lv = p.list_val + static_cast<size_t>(slot) * kTkStore;
  bool found = false;
  float xd = 0.f;
  for (int j = lane; j < cut; j += 32) {
    const int idx = static_cast<int>(0xffffffffu - static_cast<uint32_t>(sk[j] >> 32));
    const float x = key_logit(static_cast<uint32_t>(sk[j] & 0xffffffffull));
    li[j] = idx;
    lv[j] = x;
    if (idx == dtok) {
      found = true;
      xd = x;
    }
  }
  // the logit of the row's draft token if it was kept (indices are distinct:
  // at most one lane finds it)
  const unsigned fm = __ballot_sync(0xffffffffu, found);
  if (fm == 0u) {
    if (lane == 0) p.rowd[slot] = make_float2(0.f, 0.f);
  } else if (lane == __ffs(fm) - 1) {
    p.rowd[slot] = make_float2(xd, 1.f);
  }
  if (lane == 0) p.rowtk[slot] = make_float4(__int_as_float(cut), mk, lse2, __int_as_float(argmax));
}

template <typename T>
__global__ void __launch_bounds__(kTkThreads, 2) topk_select_kernel(const __grid_constant__ TopkParams p) {
  constexpr int P = Elt<T>::kPerVec;
  // hist (the radix select's per-warp histograms) is also the block-maximum
  // keys while K's superset is gathered, and the sort's scratch afterwards
  __shared__ __align__(16) int hist[kTkWarps * 256];
  __shared__ unsigned long long sk[kTkStore];
  __shared__ uint16_t qlist[kTkCollectMaxBlocks];
  __shared__ int hist256[256];
  __shared__ F2 s_wtot[kTkWarps];
  __shared__ int s_val[2], s_w[kTkWarps];
  __shared__ int s_digit, s_remaining, s_count, s_cut;
  static_assert(kTkWarps * 256 * sizeof(int) >= kTkCollectMaxBlocks * sizeof(uint32_t), "block-maximum keys");
  static_assert(kTkWarps * 256 * sizeof(int) >= kTkStore * sizeof(unsigned long long), "sort scratch");
  unsigned long long* sort_tmp = reinterpret_cast<unsigned long long*>(hist);
  grid_dep_launch();
  const int g = p.gamma, slots = 2 * g + 1;
  const int slot = blockIdx.x, b = slot / slots, t = slot - b * slots;
  // inputs of the call, read before the wait for the row reducer
  const bool greedy = seq_is_greedy(p.temperature, b);
  const float temp = p.temperature[b];
  // the draft token this row is checked against (target row t < gamma and
  // draft row t - gamma - 1 both check d_{t+1})
  const int dtok = (t == g) ? -1 : p.draft_tokens[b * g + (t < g ? t : t - g - 1)];
  grid_dep_wait();  // the row reducer's block maxima
  if (t > g && greedy) return;  // greedy sequences read no draft rows
  const void* row = (t <= g) ? static_cast<const void*>(static_cast<const T*>(p.target) +
                                                        (static_cast<size_t>(b) * (g + 1) + t) * p.V)
                             : static_cast<const void*>(static_cast<const T*>(p.draft) +
                                                        (static_cast<size_t>(b) * g + (t - g - 1)) * p.V);
  const int k = greedy ? 1 : min(p.top_k, p.V);

  // ---- K (or a superset of it) into shared memory ----
  // Usually from the block maxima.  Without them, or if that list is not
  // usable (fewer than k entries cannot happen; more than kTkStore can), a
  // threshold from a sample (its rank-s largest entry sits above about 16 s
  // entries of the row; s = k/8 + 8, about 2k + 128, capped so that 16 s
  // stays well inside the kept list), then the entries reaching it; if that
  // misses too, the exact radix select over the whole row.
  const TkRange<T> full{p.V / P, false}, smp{p.V / P, true};
  const int srank = min(k / 8 + 8, (kTkStore * 4 / 5) / 16);
  uint32_t prefix = 0, pmask = 0;
  int count = -1;
  // (with k at least the number of blocks the bound would keep every logit)
  if (p.submax != nullptr && k < p.cpr * kVecPerLane && p.cpr * kVecPerLane <= kTkCollectMaxBlocks) {
    count = tk_gather_blocks<T>(p, slot, row, k, reinterpret_cast<uint32_t*>(hist), qlist, hist256, s_val, s_w, sk,
                                &s_count);
    if (count < k || count > kTkStore) count = -1;
    __syncthreads();
  }
  if (count < 0 && p.V >= 4096) {
    // a miss gives the row's true count for that rank: the next rank is
    // scaled toward the middle of [k, kTkStore] (two more tries at most)
    int sr = srank;
#pragma unroll 1
    for (int attempt = 0; attempt < 3 && sr >= 1 && sr <= smp.count(); ++attempt) {
      tk_radix_select<T>(row, smp, sr, hist, &s_digit, &s_remaining, &prefix, &pmask);
      const int c = tk_collect<T>(row, p.V, prefix, pmask, sk, &s_count);
      __syncthreads();
      if (c >= k && c <= kTkStore) {
        count = c;
        break;
      }
      const int want = (k + kTkStore) / 2;
      const int next = static_cast<int>(static_cast<long long>(sr) * want / max(c, 1));
      sr = (next != sr) ? next : (c > kTkStore ? sr - 1 : sr + 1);
    }
  }
  if (count < 0) {
    tk_radix_select<T>(row, full, k, hist, &s_digit, &s_remaining, &prefix, &pmask);
    count = tk_collect<T>(row, p.V, prefix, pmask, sk, &s_count);
  }
  if (count > kTkStore) {  // more tied entries than the kept list holds
    if (threadIdx.x == 0) atomicOr(p.status, kStatusTopkOverflow);
    count = kTkStore;
  }
  if (count <= kTkWarpList) {  // block-uniform: a short list is finished by warp 0
    if (threadIdx.x < 32) tk_finish_warp(p, slot, k, count, greedy, temp, dtok, sk, sort_tmp);
    return;
  }
  tk_sort_keys_desc(sk, count, sort_tmp);  // logit descending, index ascending
  {
    // K: the entries whose key reaches the k-th largest (the collection may
    // hold a superset); ties with the k-th stay
    const uint32_t kth = static_cast<uint32_t>(sk[min(k, count) - 1] >> 32);
    if (threadIdx.x == 0) s_cut = count;
    __syncthreads();
    for (int j = k + threadIdx.x; j < count; j += kTkThreads)
      if (static_cast<uint32_t>(sk[j] >> 32) < kth) atomicMin(&s_cut, j);
    __syncthreads();
    count = s_cut;
    __syncthreads();
  }
  const int argmax = static_cast<int>(0xffffffffu - static_cast<uint32_t>(sk[0] & 0xffffffffull));
  if (greedy) {
    if (threadIdx.x == 0) p.rowtk[slot] = make_float4(__int_as_float(0), kNegHuge, 0.f, __int_as_float(argmax));
    return;
  }

  // ---- softmax over K, the top-p cut, the normaliser of K' ----
  const float ks = kLog2e / temp;
  const float mk = key_logit(static_cast<uint32_t>(sk[0] >> 32)) * ks;
  float e[4];
  uint32_t kj[4];
  F2 my = f2_from(0.f);
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // this thread's entries 4t .. 4t+3 (count <= 2048)
    const int j = 4 * threadIdx.x + q;
    kj[q] = (j < count) ? static_cast<uint32_t>(sk[j] >> 32) : 0u;
    e[q] = (j < count) ? ex2(fmaf(key_logit(kj[q]), ks, -mk)) : 0.f;
    my = f2_add(my, f2_from(e[q]));
  }
  const int jprev = 4 * static_cast<int>(threadIdx.x) - 1;  // the entry before this thread's first
  const uint32_t kprev = (jprev >= 0 && jprev < count) ? static_cast<uint32_t>(sk[jprev] >> 32) : 0xffffffffu;
  F2 S;
  const F2 incl = tk_block_scan(my, s_wtot, &S);
  if (threadIdx.x == 0) s_cut = count;
  __syncthreads();
  if (p.top_p < 1.f) {
    const F2 thr = f2_mul_f(S, p.top_p);
    F2 run = f2_sub(incl, my);  // mass of the entries before this thread's first
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = 4 * threadIdx.x + q;
      if (j < count) {
        const bool start = (j == 0) || (kj[q] != (q == 0 ? kprev : kj[q - 1]));
        // the group starting here is dropped once the mass above it reaches top_p
        if (start && !f2_gt(thr, run)) atomicMin(&s_cut, j);
        run = f2_add(run, f2_from(e[q]));
      }
    }
  }
  __syncthreads();
  const int cut = s_cut;
  F2 my2 = f2_from(0.f);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (4 * threadIdx.x + q < cut) my2 = f2_add(my2, f2_from(e[q]));
  F2 S2;
  tk_block_scan(my2, s_wtot, &S2);
  const float lse2 = log2f(S2.hi + S2.lo);

  // ---- K' re-sorted by vocabulary index, written out ----
  unsigned long long mine[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = 4 * threadIdx.x + q;
    mine[q] = 0ull;
    if (j < cut) {
      const uint32_t idx = 0xffffffffu - static_cast<uint32_t>(sk[j] & 0xffffffffull);
      mine[q] = (static_cast<unsigned long long>(0xffffffffu - idx) << 32) | kj[q];
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = 4 * threadIdx.x + q;
    if (j < cut) sk[j] = mine[q];
  }
  __syncthreads();
  tk_sort_keys_desc(sk, cut, sort_tmp);  // index ascending
  int* li = p.list_idx + static_cast<size_t>(slot) * kTkStore;
  float* lv = p.list_val + static_cast<size_t>(slot) * kTkStore;
  // the logit of the row's draft token if it was kept
  if (threadIdx.x == 0) p.rowd[slot] = make_float2(0.f, 0.f);
  __syncthreads();
  for (int j = threadIdx.x; j < cut; j += kTkThreads) {
    const int idx = static_cast<int>(0xffffffffu - static_cast<uint32_t>(sk[j] >> 32));
    const float x = key_logit(static_cast<uint32_t>(sk[j] & 0xffffffffull));
    li[j] = idx;
    lv[j] = x;
    if (idx == dtok) p.rowd[slot] = make_float2(x, 1.f);
  }
  if (threadIdx.x == 0) p.rowtk[slot] = make_float4(__int_as_float(cut), mk, lse2, __int_as_float(argmax));
}

struct TopkTailParams {
  TopkParams tk;
  DecideParams dp;
  const float* u_resample;
};

// Position of vocabulary index x in an ascending list of n entries (shared
// memory), or -1.
__device__ __forceinline__ int tk_find(const int* li, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int v = li[mid];
    if (v == x) return mid;
    if (v < x) lo = mid + 1;
    else hi = mid - 1;
  }
  return -1;
}

template <typename T>
__global__ void __launch_bounds__(kTkThreads, 1) topkp_tail_kernel(const __grid_constant__ TopkTailParams p) {
  __shared__ float4 rt[2 * 31 + 1];
  __shared__ float2 rd[2 * 31 + 1];
  __shared__ int sq_idx[kTkStore];
  __shared__ float sq_val[kTkStore];
  __shared__ F2 s_wtot[kTkWarps];
  __shared__ int s_n, s_first, s_lastnz;
  const TopkParams& tk = p.tk;
  const DecideParams& dp = p.dp;
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = dp.gamma, slots = 2 * g + 1;
  const bool greedy = seq_is_greedy(dp.temperature, b);
  // inputs of the call, read before the wait for the select kernel
  const float ks = greedy ? 0.f : kLog2e / dp.temperature[b];
  const float u_res = p.u_resample[b];
  int d = -1;
  float u_acc = 0.f;
  if (warp == 0 && lane < g) {
    d = dp.draft_tokens[b * g + lane];
    u_acc = dp.u_accept[b * g + lane];
  }
  grid_dep_wait();
  for (int r = threadIdx.x; r < (greedy ? g + 1 : slots); r += kTkThreads) {
    rt[r] = __ldcg(tk.rowtk + b * slots + r);
    rd[r] = __ldcg(tk.rowd + b * slots + r);
  }
  __syncthreads();
  auto list_idx = [&](int r) { return tk.list_idx + static_cast<size_t>(b * slots + r) * kTkStore; };
  auto list_val = [&](int r) { return tk.list_val + static_cast<size_t>(b * slots + r) * kTkStore; };
  auto count_of = [&](int r) { return __float_as_int(rt[r].x); };

  // ---- decision: one lane per draft position ----
  if (warp == 0) {
    bool acc = false;
    float pp = 0.f, qq = 0.f;
    if (lane < g) {
      const bool valid = d >= 0 && d < dp.V;
      if (!valid) atomicOr(dp.status, kStatusBadToken);
      if (valid && greedy) {
        acc = (d == __float_as_int(rt[lane].w));
      } else if (valid) {
        const float4 rp = rt[lane], rq = rt[g + 1 + lane];
        const float2 dp_ = rd[lane], dq_ = rd[g + 1 + lane];  // {logit of d, kept}
        const bool hp = dp_.y > 0.f, hq = dq_.y > 0.f;
        pp = hp ? ex2(fmaf(dp_.x, ks, -rp.y) - rp.z) : 0.f;
        qq = hq ? ex2(fmaf(dq_.x, ks, -rq.y) - rq.z) : 0.f;
        float rho;
        if (!hq) rho = INFINITY;      // q'(d) = 0: accepted
        else if (!hp) rho = 0.f;      // p'(d) = 0, q'(d) > 0: rejected
        else rho = ex2((dp_.x - dq_.x) * ks - (rp.y - rq.y) - (rp.z - rq.z));
        acc = u_acc < rho;
      }
    }
    const unsigned rej = ~__ballot_sync(0xffffffffu, acc) & ((1u << g) - 1u);
    const int n = rej ? (__ffs(rej) - 1) : g;
    if (lane <= g) {
      int tok = -1;
      if (lane < n) tok = d;
      else if (lane == n && greedy) tok = __float_as_int(rt[n].w);
      dp.out_tokens[b * (g + 1) + lane] = tok;
      if (dp.out_debug != nullptr) {
        constexpr float kLn2 = 0.6931471805599453f;
        const float nan = __int_as_float(0x7fc00000);
        float4 dbg = make_float4(nan, nan, nan, nan);
        if (!greedy) {
          const float Lp = (rt[lane].y + rt[lane].z) * kLn2;
          dbg = (lane < g) ? make_float4(pp, qq, Lp, (rt[g + 1 + lane].y + rt[g + 1 + lane].z) * kLn2)
                           : make_float4(0.f, 0.f, Lp, 0.f);
        }
        reinterpret_cast<float4*>(dp.out_debug)[b * (g + 1) + lane] = dbg;
      }
    }
    if (lane == 0) {
      dp.out_num[b] = n;
      s_n = n;
      s_first = INT_MAX;
      s_lastnz = -1;
    }
  }
  __syncthreads();
  if (greedy) return;

  // ---- the draw over the kept list of row n (residual) or gamma (bonus) ----
  const int n = s_n;
  const bool residual = n < g;
  const int r = residual ? n : g;
  const int cnt = count_of(r);
  const int* li = list_idx(r);
  const float* lv = list_val(r);
  const float4 rp = rt[r];
  const float4 rq = residual ? rt[g + 1 + n] : make_float4(0.f, 0.f, 0.f, 0.f);
  const float invSp = ex2(-rp.z), invSq = ex2(-rq.z);
  const int cq = residual ? count_of(g + 1 + n) : 0;
  // this thread's entries 4t .. 4t+3 of row r's list (ascending vocabulary
  // index), loaded while the draft row's list is staged
  int ix[4];
  float lx[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = 4 * threadIdx.x + q;
    ix[q] = (j < cnt) ? __ldcg(li + j) : -1;
    lx[q] = (j < cnt) ? __ldcg(lv + j) : 0.f;
  }
  if (residual) {  // the draft row's kept list, searched from shared memory
    for (int j = threadIdx.x; j < cq; j += kTkThreads) {
      sq_idx[j] = __ldcg(list_idx(g + 1 + n) + j);
      sq_val[j] = __ldcg(list_val(g + 1 + n) + j);
    }
    __syncthreads();
  }
  float w[4], wp[4];
  F2 my = f2_from(0.f), myp = f2_from(0.f);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = 4 * threadIdx.x + q;
    w[q] = wp[q] = 0.f;
    if (j < cnt) {
      wp[q] = ex2(fmaf(lx[q], ks, -rp.y)) * invSp;
      w[q] = wp[q];
      if (residual) {
        const int iq = tk_find(sq_idx, cq, ix[q]);
        const float qv = iq >= 0 ? ex2(fmaf(sq_val[iq], ks, -rq.y)) * invSq : 0.f;
        w[q] = fmaxf(0.f, wp[q] - qv);
      }
    }
    my = f2_add(my, f2_from(w[q]));
    myp = f2_add(myp, f2_from(wp[q]));
  }
  F2 Z;
  F2 incl = tk_block_scan(my, s_wtot, &Z);
  if (residual && !(Z.hi > 0.f)) {
    // Z == 0 cannot happen in exact arithmetic; if rounding produces it, draw from p'_n
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = wp[q];
    my = myp;
    incl = tk_block_scan(my, s_wtot, &Z);
  }
  const F2 target = f2_mul_f(Z, u_res);
  if (f2_gt(incl, target)) atomicMin(&s_first, static_cast<int>(threadIdx.x));
  int last_nz = -1;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (w[q] > 0.f) last_nz = 4 * threadIdx.x + q;
  if (last_nz >= 0) atomicMax(&s_lastnz, last_nz);
  __syncthreads();
  if (threadIdx.x == static_cast<unsigned>(s_first)) {
    F2 run = f2_sub(incl, my);
    int j = -1;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      run = f2_add(run, f2_from(w[q]));
      if (j < 0 && f2_gt(run, target)) j = 4 * threadIdx.x + q;
    }
    if (j < 0) j = last_nz;  // rounding inside the thread: its last nonzero entry
    if (j < 0) j = 4 * threadIdx.x;  // (the crossing thread always holds weight; kept in bounds regardless)
    int tok = -1;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (4 * static_cast<int>(threadIdx.x) + q == j) tok = ix[q];
    dp.out_tokens[b * (g + 1) + n] = tok >= 0 ? tok : __ldcg(li + j);
  } else if (threadIdx.x == 0 && s_first == INT_MAX) {
    // beyond the total (rounding): the last entry of nonzero weight
    const int j = s_lastnz < 0 ? 0 : s_lastnz;
    dp.out_tokens[b * (g + 1) + n] = cnt > 0 ? __ldcg(li + j) : 0;
  }
}

}  // namespace specv
