// rowstats.cuh — the vocab-row reducer.
//
// One pass over every logits row the verify step needs.  For each chunk of CE
// consecutive vocabulary entries (4 KB of logits) it produces a partial:
//   sampled rows (target and draft rows of sequences with T > 0):
//     M = max x, mk = fl(M*ks), s = sum 2^(fma(x, ks, -mk)), ks = log2(e)/T
//   greedy target rows: M and the lowest index holding it (no exponentials)
// Greedy draft rows are not read at all.
//
// The temperature softmax with a log-sum-exp reduction is the quantity
// "第 8 章 投机解码：一次前向，验证好几个字" (为什么输出不会变) requires to be applied
// identically to draft and target; the argmax is the greedy check of
// "自投机解码：层跳过与拒绝采样实现大模型推理加速" §3.1.
//
// Design (GB300).  Every warp owns whole work items (row, chunk), dealt to
// warps round-robin in sequence-major order, so no warp ever waits on
// another.  A chunk is 256 16-byte vectors: each lane holds 8 of them in
// registers and reduces them in two branch-free passes — the chunk maximum
// (packed bf16 max for bf16 input), then the exponentials against that fixed
// maximum — followed by one warp reduction.  Two ways to bring a chunk in:
//   kLdg  direct 128-bit global loads, 32 warps per SM keep ~128 KB in flight
//         (the default: measured fastest on GB300);
//   kTma  each warp streams its own chunks with 1-D bulk copies
//         (cp.async.bulk on the TMA engine) into a private 3-stage
//         shared-memory ring guarded by one mbarrier per stage.
// A probe of both on the bench workload measured 6.36 TB/s for direct loads
// against 5.5 TB/s for bulk-copy staging, so kLdg is the default; kTma is
// kept, selectable, and tested.
#pragma once

#include <cfloat>
#include <cuda_bf16.h>

#include "common.cuh"

namespace specv {

constexpr int kRowWarps = 16;                 // warps per CTA
constexpr int kRowThreads = kRowWarps * 32;   // 512
// Streaming 16-byte load of logits read exactly once: through the read-only
// path without allocating in L1 (no reuse there; measured 26.2 -> 25.5 us per
// launch on 151 MB).
__device__ __forceinline__ uint4 ld_stream(const uint4* a) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(a));
  return r;
}

constexpr int kVecPerLane = 8;                // 8 x 16 B per lane = 4 KB per chunk
constexpr int kChunkBytes = 32 * kVecPerLane * 16;
constexpr int kTmaStages = 3;                 // per-warp ring depth (kTma)
constexpr uint32_t kTmaRingBytes = kRowWarps * kTmaStages * kChunkBytes;  // 192 KB

enum RowMode { kRowSkip = 0, kRowArgmax = 1, kRowFull = 2 };
enum LoadPath { kLdg = 0, kTma = 1 };

struct RowStatsParams {
  const void* target;        // [B, gamma+1, V]
  const void* draft;         // [B, gamma, V] or nullptr (no dense draft rows: greedy or sparse drafts)
  const float* temperature;  // [B] or nullptr (every sequence greedy)
  float4* partials;          // [B*(2*gamma+1)*cpr] {M, s, argmax bits, mk}
  int* status;
  int B, gamma, V, CE, cpr;
  int draft_only;  // skip the target rows (their statistics come from the lm_head epilogue)
  float* submax;   // [slots*cpr*kVecPerLane] with kSubMax: the maxima of each chunk's kVecPerLane
                   // blocks of 32 vectors (the top-k / top-p collection bound)
  int debug;       // bit 0: forced-timeout self-test
};

// Row slot t of sequence b: t <= gamma is target row t, t > gamma is draft row
// t-gamma-1.
__device__ __forceinline__ int row_mode(const RowStatsParams& p, int b, int t) {
  const bool greedy = (p.temperature == nullptr) || seq_is_greedy(p.temperature, b);
  if (t <= p.gamma) return p.draft_only ? kRowSkip : (greedy ? kRowArgmax : kRowFull);
  return (greedy || p.draft == nullptr) ? kRowSkip : kRowFull;
}

template <typename T>
__device__ __forceinline__ const uint8_t* row_ptr(const RowStatsParams& p, int b, int t) {
  if (t <= p.gamma)
    return reinterpret_cast<const uint8_t*>(p.target) +
           (static_cast<size_t>(b) * (p.gamma + 1) + t) * p.V * sizeof(T);
  return reinterpret_cast<const uint8_t*>(p.draft) +
         (static_cast<size_t>(b) * p.gamma + (t - p.gamma - 1)) * p.V * sizeof(T);
}

// A 16-byte vector of -inf logits (pads the ragged end of a row).
template <typename T>
__device__ __forceinline__ uint4 neg_inf_vec();
template <>
__device__ __forceinline__ uint4 neg_inf_vec<float>() {
  return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
}
template <>
__device__ __forceinline__ uint4 neg_inf_vec<__nv_bfloat16>() {
  return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
}

// Maximum of the 4 or 8 logits in a 16-byte vector (fp32 result).
template <typename T>
__device__ __forceinline__ float vec_max(const uint4& v);
template <>
__device__ __forceinline__ float vec_max<float>(const uint4& v) {
  return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
               fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}
template <>
__device__ __forceinline__ float vec_max<__nv_bfloat16>(const uint4& v) {
  const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.x),
                                   *reinterpret_cast<const __nv_bfloat162*>(&v.y));
  const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.z),
                                   *reinterpret_cast<const __nv_bfloat162*>(&v.w));
  const __nv_bfloat162 c = __hmax2(a, b);
  const uint32_t w = *reinterpret_cast<const uint32_t*>(&c);
  float lo, hi;
  bf16x2_unpack(w, lo, hi);
  return fmaxf(lo, hi);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Sampled row chunk in registers: pass 1 the maximum, pass 2 the exponential
// sum against it.  Padding vectors hold -inf and contribute nothing.
template <typename T>
__device__ __forceinline__ float4 reduce_full(const uint4 (&v)[kVecPerLane], float ks) {
  constexpr int P = Elt<T>::kPerVec;
  float mx[kVecPerLane];
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) mx[j] = vec_max<T>(v[j]);
#pragma unroll
  for (int w = kVecPerLane / 2; w > 0; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) mx[j] = fmaxf(mx[j], mx[j + w]);
  const float M = warp_max(mx[0]);
  if (!(M > -FLT_MAX)) return make_float4(M, 0.f, __int_as_float(-1), kNegHuge);  // all -inf
  const float mk = M * ks;
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    float x[P];
    Elt<T>::unpack(v[j], x);
    float e[P];
#pragma unroll
    for (int k = 0; k < P; ++k) e[k] = ex2(fmaf(x[k], ks, -mk));
    if constexpr (P == 8) {
      s0 += e[0] + e[1];
      s1 += e[2] + e[3];
      s2 += e[4] + e[5];
      s3 += e[6] + e[7];
    } else {
      s0 += e[0];
      s1 += e[1];
      s2 += e[2];
      s3 += e[3];
    }
  }
  const float s = warp_sum((s0 + s1) + (s2 + s3));
  return make_float4(M, s, __int_as_float(-1), mk);
}

// Greedy row chunk in registers: the maximum and the lowest index holding it.
// Lane l holds chunk vectors l, l+32, ..., so its vectors ascend with j.
template <typename T>
__device__ __forceinline__ float4 reduce_argmax(const uint4 (&v)[kVecPerLane], int base, int lane) {
  constexpr int P = Elt<T>::kPerVec;
  float m = -FLT_MAX;
  int idx = -1;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    float x[P];
    Elt<T>::unpack(v[j], x);
    float vm = x[0];
#pragma unroll
    for (int k = 1; k < P; ++k) vm = fmaxf(vm, x[k]);
    int e = P - 1;
#pragma unroll
    for (int k = P - 1; k >= 0; --k) e = (x[k] == vm) ? k : e;
    const bool gt = vm > m;  // strict: an earlier vector keeps a tie
    idx = gt ? base + (lane + 32 * j) * P + e : idx;
    m = gt ? vm : m;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, off);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
    if (om > m || (om == m && static_cast<unsigned>(oi) < static_cast<unsigned>(idx))) {
      m = om;
      idx = oi;
    }
  }
  return make_float4(m, 0.f, __int_as_float(idx), kNegHuge);
}

// Walks the (row slot, chunk) items of one warp: item gw, gw + nw, gw + 2nw, ...
struct ItemIter {
  int slot, chunk, dq, dr, cpr;
  __device__ __forceinline__ void init(int gw, int nw, int cpr_) {
    cpr = cpr_;
    slot = gw / cpr;
    chunk = gw - slot * cpr;
    dq = nw / cpr;
    dr = nw - dq * cpr;
  }
  __device__ __forceinline__ void advance() {
    chunk += dr;
    slot += dq;
    if (chunk >= cpr) {
      chunk -= cpr;
      ++slot;
    }
  }
};

struct Item {
  const uint4* src;
  int slot, chunk, mode, nvec;
  float ks;
};

// Advance `it` to the next item that must be read; false when none is left.
template <typename T>
__device__ __forceinline__ bool next_live(const RowStatsParams& p, ItemIter& it, int n_slots, Item& out) {
  const int slots = 2 * p.gamma + 1;
  while (it.slot < n_slots) {
    const int b = it.slot / slots, t = it.slot - b * slots;
    const int mode = row_mode(p, b, t);
    if (mode != kRowSkip) {
      const int len = min(p.CE, p.V - it.chunk * p.CE);
      out.src = reinterpret_cast<const uint4*>(row_ptr<T>(p, b, t) +
                                               static_cast<size_t>(it.chunk) * p.CE * sizeof(T));
      out.slot = it.slot;
      out.chunk = it.chunk;
      out.mode = mode;
      out.nvec = len / Elt<T>::kPerVec;
      out.ks = (mode == kRowFull) ? kLog2e / p.temperature[b] : 0.f;
      it.advance();
      return true;
    }
    it.advance();
  }
  return false;
}

template <typename T, bool kSubMax>
__device__ __forceinline__ void finish_item(const RowStatsParams& p, const Item& d,
                                            const uint4 (&v)[kVecPerLane], int lane) {
  const float4 r = (d.mode == kRowFull) ? reduce_full<T>(v, d.ks)
                                        : reduce_argmax<T>(v, d.chunk * p.CE, lane);
  if (lane == 0 && in_bounds(d.slot >= 0 && d.slot < p.B * (2 * p.gamma + 1) && d.chunk >= 0 && d.chunk < p.cpr,
                             p.status))
    p.partials[static_cast<size_t>(d.slot) * p.cpr + d.chunk] = r;
  if constexpr (kSubMax) {
    // block j of the chunk is vector slot j of every lane (32 consecutive
    // vectors).  A warp reduce-scatter: each exchange halves the values a
    // lane holds, so the 8 maxima take 4 + 2 + 1 + 1 + 1 shuffles; lane l
    // ends with block ((l >> 4) & 1) * 4 + ((l >> 3) & 1) * 2 + ((l >> 2) & 1).
    static_assert(kVecPerLane == 8, "the reduce-scatter below is written for 8 blocks");
    float m8[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) m8[j] = vec_max<T>(v[j]);
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
    float m4[4], m2[2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float keep = h16 ? m8[q + 4] : m8[q], give = h16 ? m8[q] : m8[q + 4];
      m4[q] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 16));
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float keep = h8 ? m4[q + 2] : m4[q], give = h8 ? m4[q] : m4[q + 2];
      m2[q] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 8));
    }
    float m = fmaxf(h4 ? m2[1] : m2[0], __shfl_xor_sync(0xffffffffu, h4 ? m2[0] : m2[1], 4));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    if ((lane & 3) == 0) {
      const int j = (h16 ? 4 : 0) + (h8 ? 2 : 0) + (h4 ? 1 : 0);
      p.submax[(static_cast<size_t>(d.slot) * p.cpr + d.chunk) * kVecPerLane + j] = m;
    }
  }
}

template <typename T, int kPath, bool kSubMax = false>
__global__ void __launch_bounds__(kRowThreads, (kPath == kLdg) ? 2 : 1)
    rowstats_kernel(const RowStatsParams p) {
  extern __shared__ __align__(128) uint8_t ring[];  // kTma only
  __shared__ __align__(8) uint64_t bar[kRowWarps * kTmaStages];
  __shared__ __align__(8) uint64_t never_bar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_launch();  // let the accept kernel's launch overlap this one
  grid_dep_wait();    // the logits and the workspace may come from the previous grid

  if (p.debug & 1) {  // self-test: a wait nobody can satisfy must end by itself
    if (threadIdx.x == 0) {
      mbar_init(&never_bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (lane == 0) mbar_wait(&never_bar, 0, p.status, kWaitLimitCyclesShort);
    return;
  }

  const int n_slots = p.B * (2 * p.gamma + 1);
  ItemIter it;
  it.init(blockIdx.x * kRowWarps + warp, gridDim.x * kRowWarps, p.cpr);
  Item d;

  if constexpr (kPath == kLdg) {
    while (next_live<T>(p, it, n_slots, d)) {
      uint4 v[kVecPerLane];
#pragma unroll
      for (int j = 0; j < kVecPerLane; ++j) {
        const int k = lane + 32 * j;
        v[j] = (k < d.nvec) ? ld_stream(d.src + k) : neg_inf_vec<T>();
      }
      finish_item<T, kSubMax>(p, d, v, lane);
    }
  } else {
    // private ring of kTmaStages chunks per warp; lane 0 issues the copies
    uint8_t* my = ring + static_cast<size_t>(warp) * kTmaStages * kChunkBytes;
    uint64_t* mb = bar + warp * kTmaStages;
    if (lane == 0) {
      for (int s = 0; s < kTmaStages; ++s) mbar_init(&mb[s], 1);
      fence_mbar_init();
    }
    __syncwarp();
    ItemIter iss = it;  // the issue walk runs up to kTmaStages items ahead
    Item di;
    int issued = 0, consumed = 0;
    for (; issued < kTmaStages && next_live<T>(p, iss, n_slots, di); ++issued) {
      if (lane == 0) {
        const uint32_t bytes = static_cast<uint32_t>(di.nvec) * 16u;
        mbar_arrive_expect_tx(&mb[issued], bytes);
        bulk_g2s(my + issued * kChunkBytes, di.src, bytes, &mb[issued]);
      }
    }
    bool ok = true;
    while (consumed < issued) {
      next_live<T>(p, it, n_slots, d);  // the item in flight in this stage
      const int s = consumed % kTmaStages;
      const bool got = mbar_wait(&mb[s], (consumed / kTmaStages) & 1, p.status, kWaitLimitCycles);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      const uint4* sv = reinterpret_cast<const uint4*>(my + s * kChunkBytes);
      uint4 v[kVecPerLane];
#pragma unroll
      for (int j = 0; j < kVecPerLane; ++j) {
        const int k = lane + 32 * j;
        v[j] = (k < d.nvec) ? sv[k] : neg_inf_vec<T>();
      }
      ++consumed;
      __syncwarp();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (next_live<T>(p, iss, n_slots, di)) {  // refill this stage before computing
        if (lane == 0) {
          const uint32_t bytes = static_cast<uint32_t>(di.nvec) * 16u;
          mbar_arrive_expect_tx(&mb[s], bytes);
          bulk_g2s(my + s * kChunkBytes, di.src, bytes, &mb[s]);
        }
        ++issued;
      }
      finish_item<T, kSubMax>(p, d, v, lane);
    }
    if (!ok) {  // drain: copies still in flight land before the CTA exits
      for (int k = consumed; k < issued; ++k)
        if (lane == 0) mbar_wait(&mb[k % kTmaStages], (k / kTmaStages) & 1, p.status, kWaitLimitCycles);
    }
  }
}

}  // namespace specv
