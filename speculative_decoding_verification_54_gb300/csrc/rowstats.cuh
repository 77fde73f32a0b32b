// rowstats.cuh — the vocab-row reducer.
//
// One pass over every logits row the verify step needs: for each chunk of CE
// consecutive vocabulary entries it produces the online-softmax partial
// (raw max m, scaled max mk = fl(m*ks), s = sum 2^(fma(x, ks, -mk)), argmax)
// with ks = log2(e)/T.  The rows are the target rows of every sequence and
// the draft rows of sampling sequences; greedy target rows only need the
// argmax, greedy draft rows are not read at all.
//
// The temperature softmax with a log-sum-exp reduction is the quantity
// "第 8 章 投机解码：一次前向，验证好几个字" (为什么输出不会变) requires to be applied
// identically to draft and target; the argmax is the greedy check of
// "自投机解码：层跳过与拒绝采样实现大模型推理加速" §3.1.
//
// Design (GB300): a persistent grid of one CTA per SM.  One producer thread
// streams chunks with 1-D bulk copies (cp.async.bulk, TMA engine) into a ring
// of shared-memory stages guarded by full/empty mbarriers; eight consumer
// warps each own one stage at a time, read it with conflict-free 16-byte
// LDS, and fold it into per-lane partials that one warp reduction combines.
// Items (row, chunk) are dealt to CTAs round-robin in sequence-major order so
// that every CTA streams the same number of bytes.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace specv {

constexpr int kRowWarps = 8;                      // consumer warps
constexpr int kRowThreads = (kRowWarps + 1) * 32;  // + one producer warp
constexpr int kMaxStages = 64;
constexpr uint32_t kRingBytes = 192 * 1024;

enum RowMode { kRowSkip = 0, kRowArgmax = 1, kRowFull = 2 };

struct RowStatsParams {
  const void* target;        // [B, gamma+1, V]
  const void* draft;         // [B, gamma, V] or nullptr (greedy entry point)
  const float* temperature;  // [B] or nullptr (every sequence greedy)
  float4* partials;          // [B*(2*gamma+1)*cpr] {m, s, idx bits, mk}
  int* status;
  int B, gamma, V, CE, cpr;
  int n_items;  // B*(2*gamma+1)*cpr
  int nstages;
  uint32_t stage_bytes;
  int debug;  // bit 0: forced-timeout self-test
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

// Fold one staged chunk into a warp partial.
template <typename T, bool kFull>
__device__ __forceinline__ float4 reduce_chunk(const uint4* v, int nvec, int base, float ks,
                                               int lane) {
  constexpr int P = Elt<T>::kPerVec;
  float m = -FLT_MAX, mk = kNegHuge, s0 = 0.f, s1 = 0.f;
  int idx = -1;
#pragma unroll 4
  for (int i = lane; i < nvec; i += 32) {
    float x[P];
    Elt<T>::unpack(v[i], x);
    float vm = x[0];
#pragma unroll
    for (int j = 1; j < P; ++j) vm = fmaxf(vm, x[j]);
    if (vm > m) {  // new running maximum: rare after the first vectors
      int j = 0;
      while (j < P - 1 && x[j] != vm) ++j;
      idx = base + i * P + j;
      if (kFull) {
        const float nmk = vm * ks;
        const float sc = ex2(mk - nmk);
        s0 *= sc;
        s1 *= sc;
        mk = nmk;
      }
      m = vm;
    }
    if (kFull) {
      float e[P];
#pragma unroll
      for (int j = 0; j < P; ++j) e[j] = ex2(fmaf(x[j], ks, -mk));
      if (P == 8) {
        s0 += (e[0] + e[1]) + (e[2] + e[3]);
        s1 += (e[4 % P] + e[5 % P]) + (e[6 % P] + e[7 % P]);
      } else {
        s0 += e[0] + e[1];
        s1 += e[2 % P] + e[3 % P];
      }
    }
  }
  float s = s0 + s1;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, off);
    const float omk = __shfl_xor_sync(0xffffffffu, mk, off);
    const float os = __shfl_xor_sync(0xffffffffu, s, off);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
    merge_partial(m, mk, s, idx, om, omk, os, oi);
  }
  return make_float4(m, s, __int_as_float(idx), mk);
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads, 1) rowstats_kernel(const RowStatsParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t never_bar;

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

  const int G = gridDim.x;
  if (warp == kRowWarps) {
    // ---------------- producer: one elected thread issues bulk copies -------
    if (lane != 0) return;
    uint64_t armed = 0, parity = 0;
    int live = 0;
    for (int it = blockIdx.x; it < p.n_items; it += G) {
      const int slot = it / p.cpr, c = it - slot * p.cpr;
      const int b = slot / slots, t = slot - b * slots;
      if (row_mode(p, b, t) == kRowSkip) continue;
      const int st = live % p.nstages, use = live / p.nstages;
      if (use > 0 && !mbar_wait(&empty_bar[st], (use - 1) & 1, p.status, kWaitLimitCycles)) break;
      const int len = min(p.CE, p.V - c * p.CE);
      const uint32_t bytes = static_cast<uint32_t>(len) * sizeof(T);
      mbar_arrive_expect_tx(&full_bar[st], bytes);
      bulk_g2s(ring + static_cast<size_t>(st) * p.stage_bytes,
               row_ptr<T>(p, b, t) + static_cast<size_t>(c) * p.CE * sizeof(T), bytes,
               &full_bar[st]);
      armed |= 1ull << st;
      parity = (parity & ~(1ull << st)) | (static_cast<uint64_t>(use & 1) << st);
      ++live;
    }
    // drain: every copy this CTA issued has landed before it exits
    for (int st = 0; st < p.nstages; ++st)
      if (armed >> st & 1) mbar_wait(&full_bar[st], (parity >> st) & 1, p.status, kWaitLimitCycles);
    return;
  }

  // ---------------- consumers -----------------------------------------------
  int live = 0;
  for (int it = blockIdx.x; it < p.n_items; it += G) {
    const int slot = it / p.cpr, c = it - slot * p.cpr;
    const int b = slot / slots, t = slot - b * slots;
    const int mode = row_mode(p, b, t);
    if (mode == kRowSkip) continue;
    const int st = live % p.nstages, use = live / p.nstages;
    const bool mine = (live % kRowWarps) == warp;
    ++live;
    if (!mine) continue;
    const bool ok = mbar_wait(&full_bar[st], use & 1, p.status, kWaitLimitCycles);
    if (!__all_sync(0xffffffffu, ok)) break;
    const int len = min(p.CE, p.V - c * p.CE);
    const uint4* v = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(st) * p.stage_bytes);
    const int nvec = len / Elt<T>::kPerVec;
    float4 r;
    if (mode == kRowFull) {
      const float ks = kLog2e / p.temperature[b];
      r = reduce_chunk<T, true>(v, nvec, c * p.CE, ks, lane);
    } else {
      r = reduce_chunk<T, false>(v, nvec, c * p.CE, 0.f, lane);
    }
    __syncwarp();
    if (lane == 0) {
      p.partials[static_cast<size_t>(slot) * p.cpr + c] = r;
      mbar_arrive(&empty_bar[st]);
    }
  }
}

}  // namespace specv
