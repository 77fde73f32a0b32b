// common.cuh — shared device helpers for the verify kernels (sm_103a).
//
// Inline PTX wrappers for mbarriers and 1-D bulk copies (cp.async.bulk, the
// TMA engine's untiled form), bounded waits that record a timeout in the
// workspace status word instead of hanging, and the workspace layout.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cuda/atomic>

namespace specv {

// ---------------------------------------------------------------------------
// status bits (OR-ed into the workspace status word on the device)
// ---------------------------------------------------------------------------
constexpr int kStatusTimeout = 1;
constexpr int kStatusBadToken = 2;
constexpr int kStatusTopkOverflow = 4;  // more tied entries than a truncation list holds
constexpr int kStatusLimit = 8;         // more candidates than the caller's capacity (centroid head)
constexpr int kStatusBounds = 16;       // an index failed its check (bounds-checked build only)

// Bounds checks of the debug build.  Built with -DSPEC_CHECK_BOUNDS, every
// checked index that falls outside its extent ORs kStatusBounds into the
// status word and the access it guards is skipped (no trap: the context stays
// usable and spec_verify_status reports it).  In the normal build the check
// is the constant true and costs nothing.
#ifdef SPEC_CHECK_BOUNDS
constexpr bool kCheckBounds = true;
__device__ __forceinline__ bool in_bounds(bool ok, int* status) {
  if (!ok) atomicOr(status, kStatusBounds);
  return ok;
}
#else
constexpr bool kCheckBounds = false;
__device__ __forceinline__ bool in_bounds(bool, int*) { return true; }
#endif

// wait limits in SM clock cycles (~2 GHz): about one second normally
constexpr long long kWaitLimitCycles = 2000000000LL;
constexpr long long kWaitLimitCyclesShort = 2000000LL;  // forced-timeout self-test

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegHuge = -3.0e38f;  // stands for -inf in scaled maxima

// completion counters each sit on their own 128-byte line (no atomic
// contention between sequences)
constexpr int kCounterStride = 32;

// sequence modes written by the deciding warp
constexpr int kModeGreedy = 0;    // fully decided (greedy or greedy row)
constexpr int kModeResidual = 1;  // sample position n from max(0, p_n - q_n)
constexpr int kModeBonus = 2;     // all accepted: sample the bonus from p_gamma

// ---------------------------------------------------------------------------
// workspace layout (all offsets 256-byte aligned)
// ---------------------------------------------------------------------------
struct WsHeader {
  int status;
  int pad[63];
};

struct RowStat {  // combined statistics of one logits row
  float mk;       // fl(max_raw * ks): scaled max
  int argmax;     // lowest index of the raw maximum (greedy rows)
  float lse2;     // log2 of sum_x 2^(fma(x, ks, -mk))
  int pad;
};

struct SeqState {
  int n;     // accepted drafts
  int mode;  // kMode*
  float ks;  // log2(e) / T
  int pad;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  On timeout the status word gets
// kStatusTimeout and false is returned; the caller then stops its work.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// 1-D bulk copy global -> shared, completion signalled on `bar` (bytes and both
// addresses must be multiples of 16).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before its predecessor ends; it must call
// grid_dep_wait() before reading anything the predecessor wrote.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 2^x on the MUFU unit (ex2.approx.ftz.f32).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void bf16x2_unpack(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

template <typename T>
struct Elt;
template <>
struct Elt<float> {
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  __device__ static __forceinline__ void unpack(const uint4& v, float* x) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ float load1(const void* base, size_t i) {
    return reinterpret_cast<const float*>(base)[i];
  }
};
template <>
struct Elt<__nv_bfloat16> {
  static constexpr int kPerVec = 8;
  __device__ static __forceinline__ void unpack(const uint4& v, float* x) {
    bf16x2_unpack(v.x, x[0], x[1]);
    bf16x2_unpack(v.y, x[2], x[3]);
    bf16x2_unpack(v.z, x[4], x[5]);
    bf16x2_unpack(v.w, x[6], x[7]);
  }
  __device__ static __forceinline__ float load1(const void* base, size_t i) {
    const uint16_t b = reinterpret_cast<const uint16_t*>(base)[i];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
};

// A sequence is sampled iff its temperature is a positive number.
__device__ __forceinline__ bool seq_is_greedy(const float* temperature, int b) {
  if (temperature == nullptr) return true;
  const float t = temperature[b];
  return !(t > 0.0f);
}

// The last-CTA handoff of a sequence's tail: every CTA adds one to the
// sequence's counter with an acquire-release atomic after a barrier (the
// barrier orders the CTA's writes before thread 0's release); the CTA that
// brings it to `parts` sees all of them once it has passed the next barrier,
// and resets the counter for the next call.
__device__ __forceinline__ bool last_cta_arrives(int* counter, int parts) {
  cuda::atomic_ref<int, cuda::thread_scope_device> c(*counter);
  const int old = c.fetch_add(1, cuda::memory_order_acq_rel);
  const bool last = (old == parts - 1);
  if (last) c.store(0, cuda::memory_order_relaxed);
  return last;
}

// Compensated (Neumaier) summation: s + c carries the sum to about twice the
// working precision, so fp32 suffices where fp64 would be slow on GB300.
__device__ __forceinline__ void neumaier_add(float& s, float& c, float x) {
  const float t = s + x;
  c += (fabsf(s) >= fabsf(x)) ? ((s - t) + x) : ((x - t) + s);
  s = t;
}

// Merge two online-softmax partials (raw max m, scaled max mk, sum s relative
// to 2^mk, argmax idx; idx compared unsigned so -1 never wins a tie).
__device__ __forceinline__ void merge_partial(float& m, float& mk, float& s, int& idx, float om,
                                              float omk, float os, int oidx) {
  const float nmk = fmaxf(mk, omk);
  s = s * ex2(mk - nmk) + os * ex2(omk - nmk);
  mk = nmk;
  if (om > m || (om == m && static_cast<unsigned>(oidx) < static_cast<unsigned>(idx))) idx = oidx;
  m = fmaxf(m, om);
}

}  // namespace specv
