// rowstats.cuh — the vocab-row reducer.
//
// One pass over every logits row the verify step needs.  For each chunk of CE
// consecutive vocabulary entries it produces a partial:
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
// Design (GB300): a persistent grid of one CTA per SM.  One producer thread
// streams 4 KB chunks with 1-D bulk copies (cp.async.bulk on the TMA engine)
// into a 48-stage shared-memory ring guarded by full/empty mbarriers and
// writes a small descriptor per stage.  Sixteen consumer warps take stages
// round-robin, so stage s always belongs to warp s % 16 (the stage count is a
// multiple of 16): a warp only ever waits on the next phase of a stage it
// released itself, which keeps the mbarrier parity waits unambiguous.  Each
// warp reduces its stage in two branch-free passes over shared
// memory: the chunk maximum (packed bf16 max for bf16 input), then the
// exponentials against that fixed maximum, so no per-element rescaling chain
// limits the pipeline.  Items (row, chunk) are dealt to CTAs round-robin in
// sequence-major order so every CTA streams about the same number of bytes.
#pragma once

#include <cfloat>
#include <cuda_bf16.h>

#include "common.cuh"

namespace specv {

constexpr int kRowWarps = 16;                      // consumer warps
constexpr int kRowThreads = (kRowWarps + 1) * 32;  // + one producer warp
constexpr int kMaxStages = 64;
constexpr uint32_t kRingBytes = 208 * 1024;
constexpr uint32_t kStageBytesMax = 4096;

enum RowMode { kRowSkip = 0, kRowArgmax = 1, kRowFull = 2 };

struct RowStatsParams {
  const void* target;        // [B, gamma+1, V]
  const void* draft;         // [B, gamma, V] or nullptr (greedy entry point)
  const float* temperature;  // [B] or nullptr (every sequence greedy)
  float4* partials;          // [B*(2*gamma+1)*cpr] {M, s, argmax bits, mk}
  int* status;
  int B, gamma, V, CE, cpr;
  int n_items;  // B*(2*gamma+1)*cpr
  int nstages;
  uint32_t stage_bytes;
  int debug;  // bit 0: forced-timeout self-test
};

struct StageDesc {  // written by the producer before it arms a stage
  int slot;         // row slot, or -1: no more work for the consumer
  int chunk;
  int mode;
  float ks;
};

// Row slot t of sequence b: t <= gamma is target row t, t > gamma is draft row
// t-gamma-1.
__device__ __forceinline__ int row_mode(const RowStatsParams& p, int b, int t) {
  const bool greedy = (p.draft == nullptr) || seq_is_greedy(p.temperature, b);
  if (t <= p.gamma) return greedy ? kRowArgmax : kRowFull;
  return greedy ? kRowSkip : kRowFull;
}

template <typename T>
__device__ __forceinline__ const uint8_t* row_ptr(const RowStatsParams& p, int b, int t) {
  if (t <= p.gamma)
    return reinterpret_cast<const uint8_t*>(p.target) +
           (static_cast<size_t>(b) * (p.gamma + 1) + t) * p.V * sizeof(T);
  return reinterpret_cast<const uint8_t*>(p.draft) +
         (static_cast<size_t>(b) * p.gamma + (t - p.gamma - 1)) * p.V * sizeof(T);
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

// Sampled row chunk: pass 1 the maximum, pass 2 the exponential sum against it.
template <typename T>
__device__ __forceinline__ float4 reduce_full(const uint4* v, int nvec, float ks, int lane) {
  constexpr int P = Elt<T>::kPerVec;
  float m0 = -FLT_MAX, m1 = -FLT_MAX;
  int i = lane;
  for (; i + 32 < nvec; i += 64) {
    m0 = fmaxf(m0, vec_max<T>(v[i]));
    m1 = fmaxf(m1, vec_max<T>(v[i + 32]));
  }
  if (i < nvec) m0 = fmaxf(m0, vec_max<T>(v[i]));
  const float M = warp_max(fmaxf(m0, m1));
  if (!(M > -FLT_MAX)) return make_float4(M, 0.f, __int_as_float(-1), kNegHuge);  // all -inf
  const float mk = M * ks;
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll 2
  for (i = lane; i < nvec; i += 32) {
    float x[P];
    Elt<T>::unpack(v[i], x);
    float e[P];
#pragma unroll
    for (int j = 0; j < P; ++j) e[j] = ex2(fmaf(x[j], ks, -mk));
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

// Greedy row chunk: maximum and the lowest index holding it.
template <typename T>
__device__ __forceinline__ float4 reduce_argmax(const uint4* v, int nvec, int base, int lane) {
  constexpr int P = Elt<T>::kPerVec;
  float m = -FLT_MAX;
  int vb = -1;
  for (int i = lane; i < nvec; i += 32) {
    const float vm = vec_max<T>(v[i]);
    const bool gt = vm > m;  // strict: the earliest vector keeps a tie
    m = gt ? vm : m;
    vb = gt ? i : vb;
  }
  int idx = -1;
  if (vb >= 0) {
    float x[P];
    Elt<T>::unpack(v[vb], x);
    int j = P - 1;
#pragma unroll
    for (int k = P - 1; k >= 0; --k) j = (x[k] == m) ? k : j;
    idx = base + vb * P + j;
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

template <typename T>
__global__ void __launch_bounds__(kRowThreads, 1) rowstats_kernel(const RowStatsParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t never_bar;
  __shared__ StageDesc desc[kMaxStages];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slots = 2 * p.gamma + 1;
  grid_dep_launch();  // let the accept kernel's launch overlap this one
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nstages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&never_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  if (p.debug & 1) {  // self-test: a wait nobody can satisfy must end by itself
    if (lane == 0) mbar_wait(&never_bar, 0, p.status, kWaitLimitCyclesShort);
    return;
  }

  if (warp == kRowWarps) {
    // ---------------- producer: one elected thread issues bulk copies -------
    if (lane != 0) return;
    uint64_t armed = 0, parity = 0;
    int live = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
      const int slot = it / p.cpr, c = it - slot * p.cpr;
      const int b = slot / slots, t = slot - b * slots;
      const int mode = row_mode(p, b, t);
      if (mode == kRowSkip) continue;
      const int st = live % p.nstages, use = live / p.nstages;
      if (use > 0 && !mbar_wait(&empty_bar[st], (use - 1) & 1, p.status, kWaitLimitCycles)) {
        ok = false;
        break;
      }
      const int len = min(p.CE, p.V - c * p.CE);
      const uint32_t bytes = static_cast<uint32_t>(len) * sizeof(T);
      StageDesc d;
      d.slot = slot;
      d.chunk = c;
      d.mode = mode;
      d.ks = (mode == kRowFull) ? kLog2e / p.temperature[b] : 0.f;
      desc[st] = d;
      mbar_arrive_expect_tx(&full_bar[st], bytes);
      bulk_g2s(ring + static_cast<size_t>(st) * p.stage_bytes,
               row_ptr<T>(p, b, t) + static_cast<size_t>(c) * p.CE * sizeof(T), bytes, &full_bar[st]);
      armed |= 1ull << st;
      parity = (parity & ~(1ull << st)) | (static_cast<uint64_t>(use & 1) << st);
      ++live;
    }
    // one end marker per consumer warp (each warp's next stage index)
    for (int w = 0; w < kRowWarps && ok; ++w) {
      const int st = live % p.nstages, use = live / p.nstages;
      if (use > 0 && !mbar_wait(&empty_bar[st], (use - 1) & 1, p.status, kWaitLimitCycles)) break;
      desc[st].slot = -1;
      mbar_arrive(&full_bar[st]);
      armed &= ~(1ull << st);  // the marker advanced the phase past the last copy
      ++live;
    }
    // drain: every copy this CTA issued has landed before it exits
    for (int st = 0; st < p.nstages; ++st)
      if (armed >> st & 1) mbar_wait(&full_bar[st], (parity >> st) & 1, p.status, kWaitLimitCycles);
    return;
  }

  // ---------------- consumers: warp w takes stage indices w, w+16, ... -------
  for (int k = warp;; k += kRowWarps) {
    const int st = k % p.nstages, use = k / p.nstages;
    const bool ok = mbar_wait(&full_bar[st], use & 1, p.status, kWaitLimitCycles);
    if (!__all_sync(0xffffffffu, ok)) break;
    const StageDesc d = desc[st];
    if (d.slot < 0) break;
    const int len = min(p.CE, p.V - d.chunk * p.CE);
    const uint4* v = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(st) * p.stage_bytes);
    const int nvec = len / Elt<T>::kPerVec;
    const float4 r = (d.mode == kRowFull) ? reduce_full<T>(v, nvec, d.ks, lane)
                                          : reduce_argmax<T>(v, nvec, d.chunk * p.CE, lane);
    __syncwarp();
    if (lane == 0) {
      p.partials[static_cast<size_t>(d.slot) * p.cpr + d.chunk] = r;
      mbar_arrive(&empty_bar[st]);
    }
  }
}

}  // namespace specv
