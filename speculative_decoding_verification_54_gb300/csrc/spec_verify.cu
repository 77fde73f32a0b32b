// spec_verify.cu — host side of libspecverify: argument checks, workspace
// layout and kernel launches behind the C ABI declared in spec_verify.h.
//
// Launch chain of one call (all on the caller's stream):
//   rowstats  chunk partials of every row the call needs (argmax for greedy
//             target rows, softmax statistics for sampled rows)
//   tail      per sequence: row combine, acceptance decision, and for sampled
//             sequences the residual / bonus chunk masses and the draw
// The tail kernel is launched with programmatic stream serialization so its
// launch latency overlaps the row reducer; it waits for the reducer's results
// with griddepcontrol.wait before reading them.
//
// With the fused lm_head (spec_verify_lmhead_sample) the chain is
//   rowstats (draft rows only) -> lmhead (tcgen05 GEMM + statistics epilogue)
//   -> lm_decide -> lm_tail,
// every launch after the first with programmatic stream serialization.
#include <cuda.h>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "centroid.cuh"
#include "common.cuh"
#include "decide.cuh"
#include "lmhead.cuh"
#include "lmtail.cuh"
#include "rowstats.cuh"
#include "sample.cuh"
#include "sparse.cuh"
#include "spec_verify.h"
#include "tc.cuh"
#include "topkp.cuh"

using namespace specv;

namespace {

constexpr int kMinChunk = 1024;  // smallest vocab chunk (elements)
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int sms = 0;
  int path = kLdg;     // row-reducer load path (SPECV_ROW_LOADS=tma selects kTma)
  int lm_max_dyn = 0;  // dynamic shared memory the lm_head kernel may use
  bool ready = false;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;
int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SPEC_ERR_CUDA;
    const int smem = static_cast<int>(kTmaRingBytes);
    if (cudaFuncSetAttribute(rowstats_kernel<float, kTma>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess ||
        cudaFuncSetAttribute(rowstats_kernel<__nv_bfloat16, kTma>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, lmhead_kernel<2>) != cudaSuccess)
      return SPEC_ERR_CUDA;
    d.lm_max_dyn = optin - static_cast<int>(fa.sharedSizeBytes);
    if (cudaFuncSetAttribute(lmhead_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, d.lm_max_dyn) !=
            cudaSuccess ||
        cudaFuncSetAttribute(lmhead_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, d.lm_max_dyn) !=
            cudaSuccess)
      return SPEC_ERR_CUDA;
    // the centroid head: cluster keys (4 B each) and the candidate ranking
    // (candidates plus the token bitmap and its prefix) in shared memory
    if (cudaFuncSetAttribute(cluster_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kHeadMaxClusters * 4) != cudaSuccess ||
        cudaFuncSetAttribute(cand_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kHeadSortSmemBitmap)) != cudaSuccess ||
        cudaFuncSetAttribute(cluster_score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kScStages * sc_stage_bytes(kScMaxN) + 1024)) != cudaSuccess)
      return SPEC_ERR_CUDA;
    const char* env = std::getenv("SPECV_ROW_LOADS");
    d.path = (env != nullptr && std::strcmp(env, "tma") == 0) ? kTma : kLdg;
    d.ready = true;
  }
  *out = d;
  return SPEC_OK;
}

struct Layout {
  size_t header, partials, mass, tail_done, cand, total;
};

// Offsets of the workspace regions for a call with (B, gamma, V); sized for
// the smallest chunk so any chunk choice fits.
Layout layout(int B, int gamma, int V) {
  const size_t slots = static_cast<size_t>(B) * (2 * gamma + 1);
  const size_t cpr = (static_cast<size_t>(V) + kMinChunk - 1) / kMinChunk;
  Layout L;
  size_t off = 0;
  L.header = off;
  off += align_up(sizeof(WsHeader), 256);
  L.partials = off;
  off += align_up(slots * cpr * sizeof(float4), 256);
  L.mass = off;
  off += align_up(static_cast<size_t>(B) * cpr * sizeof(float), 256);
  L.tail_done = off;  // per-sequence counters: zero when no call is running
  off += align_up(static_cast<size_t>(B) * kCounterStride * sizeof(int), 256);
  L.cand = off;  // per-candidate outputs of the multi-candidate entry: tokens [B, gamma+1], counts [B]
  off += align_up(static_cast<size_t>(B) * (gamma + 2) * sizeof(int32_t), 256);
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int B, int gamma, int V) {
  if (B < 1 || B > 65535) return SPEC_ERR_INVALID_ARG;
  if (gamma < 1 || gamma > SPEC_MAX_GAMMA) return SPEC_ERR_INVALID_ARG;
  if (V < 8 || V > SPEC_MAX_VOCAB || (V % 8) != 0) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

// Chunk size: 4 KB of logits per chunk (one warp's work item), halved while
// the grid would have fewer than 2 chunks per SM, never below kMinChunk
// elements.  Halving further buys the row reducer nothing and costs the tail:
// one sequence (9 rows of 262,144 bf16) measured 13.8 us per call with
// 1,024-entry chunks (2,304 items) against 11.0 us with 2,048 (1,152 items):
// the fold and the draw's scan read half as many partials.
struct Plan {
  int CE, cpr, grid;
  size_t smem;
};

Plan make_plan_rows(int rows, int V, size_t esize, int sms, int path) {
  Plan p;
  int CE = static_cast<int>(kChunkBytes / esize);
  while (CE > kMinChunk && static_cast<long long>(rows) * ((V + CE - 1) / CE) < 2LL * sms) CE >>= 1;
  p.CE = CE;
  p.cpr = (V + CE - 1) / CE;
  const long long live_items = static_cast<long long>(rows) * p.cpr;
  const int per_sm = (path == kLdg) ? 2 : 1;  // CTAs resident per SM
  const long long want = (live_items + kRowWarps - 1) / kRowWarps;
  p.grid = static_cast<int>(want < static_cast<long long>(per_sm) * sms ? want : per_sm * sms);
  if (p.grid < 1) p.grid = 1;
  p.smem = (path == kTma) ? kTmaRingBytes : 0;
  return p;
}

Plan make_plan(int B, int gamma, int V, size_t esize, int sms, bool sampling, int path) {
  return make_plan_rows(B * (sampling ? (2 * gamma + 1) : (gamma + 1)), V, esize, sms, path);
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern k, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

struct Common {
  const void* target;
  const void* draft;
  spec_dtype dt;
  const int32_t* draft_tokens;
  const float* temperature;
  const float* u_accept;
  const float* u_resample;
  int B, gamma, V;
  int32_t* out_tokens;
  int32_t* out_num;
  float* out_debug;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  int debug;
  bool reduce_only;  // launch only the row reducer (timing / profiling)
};

template <typename T>
int run_chain(const Common& a, bool sampling) {
  const Layout L = layout(a.B, a.gamma, a.V);
  if (a.ws_bytes < L.total) return SPEC_ERR_WORKSPACE;
  DeviceInfo dev;
  if (device_info(&dev) != SPEC_OK) return SPEC_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  int* status = reinterpret_cast<int*>(ws + L.header);
  const Plan pl = make_plan(a.B, a.gamma, a.V, sizeof(T), dev.sms, sampling, dev.path);

  RowStatsParams rp = {};
  rp.target = a.target;
  rp.draft = sampling ? a.draft : nullptr;
  rp.temperature = sampling ? a.temperature : nullptr;
  rp.partials = reinterpret_cast<float4*>(ws + L.partials);
  rp.status = status;
  rp.B = a.B;
  rp.gamma = a.gamma;
  rp.V = a.V;
  rp.CE = pl.CE;
  rp.cpr = pl.cpr;
  rp.debug = a.debug;
  // programmatic launch: the reducer waits for the previous grid in the stream
  // (griddepcontrol.wait) before it reads anything, so only the launch
  // latency overlaps the predecessor's tail
  cudaError_t e;
  if (dev.path == kTma)
    e = launch_pdl(rowstats_kernel<T, kTma>, dim3(pl.grid), dim3(kRowThreads), pl.smem, a.stream, rp);
  else
    e = launch_pdl(rowstats_kernel<T, kLdg>, dim3(pl.grid), dim3(kRowThreads), 0, a.stream, rp);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (a.debug || a.reduce_only) return SPEC_OK;

  SampleParams sp;
  sp.target = a.target;
  sp.draft = rp.draft;
  sp.u_resample = a.u_resample;
  sp.partials = rp.partials;
  sp.mass = reinterpret_cast<float*>(ws + L.mass);
  sp.tail_done = reinterpret_cast<int*>(ws + L.tail_done);
  sp.B = a.B;
  sp.gamma = a.gamma;
  sp.V = a.V;
  sp.CE = pl.CE;
  sp.cpr = pl.cpr;
  DecideParams& dp = sp.dp;
  dp.target = a.target;
  dp.draft = rp.draft;
  dp.draft_tokens = a.draft_tokens;
  dp.temperature = rp.temperature;
  dp.u_accept = a.u_accept;
  dp.out_tokens = a.out_tokens;
  dp.out_num = a.out_num;
  dp.out_debug = sampling ? a.out_debug : nullptr;
  dp.status = status;
  dp.gamma = a.gamma;
  dp.V = a.V;
  // parts per sequence: as many CTAs as fit on the GPU at once (two per SM),
  // at most 16, so the tail's CTAs all start as the row reducer frees the SMs
  // (a second wave would start late) and the residual masses spread over every
  // SM; greedy calls need one (no residual pass)
  int parts = sampling ? (2 * dev.sms) / a.B : 1;
  if (parts > 16) parts = 16;
  if (parts > pl.cpr) parts = pl.cpr;
  if (parts < 1) parts = 1;
  if (launch_pdl(tail_kernel<T>, dim3(parts, a.B), dim3(kTailThreads), 0, a.stream, sp) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

int dispatch(const Common& a, bool sampling) {
  if (a.dt != SPEC_F32 && a.dt != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  const bool f32 = a.dt == SPEC_F32;
  return f32 ? run_chain<float>(a, sampling) : run_chain<__nv_bfloat16>(a, sampling);
}

// ---------------------------------------------------------------------------
// top-k / top-p chain
// ---------------------------------------------------------------------------
struct TkLayout {
  Layout base;  // header (status), the row reducer's partials
  size_t list_idx, list_val, rowtk, rowd, submax, total;
};

TkLayout tk_layout(int B, int gamma, int V) {
  TkLayout L;
  L.base = layout(B, gamma, V);
  const size_t rows = static_cast<size_t>(B) * (2 * gamma + 1);
  size_t off = L.base.total;
  L.list_idx = off;
  off += align_up(rows * kTkStore * sizeof(int), 256);
  L.list_val = off;
  off += align_up(rows * kTkStore * sizeof(float), 256);
  L.rowtk = off;
  off += align_up(rows * sizeof(float4), 256);
  L.rowd = off;
  off += align_up(rows * sizeof(float2), 256);
  L.submax = off;  // block maxima from the row reducer
  off += align_up(rows * ((static_cast<size_t>(V) + kMinChunk - 1) / kMinChunk) * kVecPerLane * sizeof(float), 256);
  L.total = off;
  return L;
}

template <typename T>
int run_topkp(const Common& a, int top_k, float top_p) {
  const TkLayout L = tk_layout(a.B, a.gamma, a.V);
  if (a.ws_bytes < L.total) return SPEC_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  TopkTailParams tp = {};
  TopkParams& k = tp.tk;
  k.target = a.target;
  k.draft = a.draft;
  k.temperature = a.temperature;
  k.list_idx = reinterpret_cast<int*>(ws + L.list_idx);
  k.list_val = reinterpret_cast<float*>(ws + L.list_val);
  k.rowtk = reinterpret_cast<float4*>(ws + L.rowtk);
  k.rowd = reinterpret_cast<float2*>(ws + L.rowd);
  k.draft_tokens = a.draft_tokens;
  k.status = reinterpret_cast<int*>(ws + L.base.header);
  k.B = a.B;
  k.gamma = a.gamma;
  k.V = a.V;
  k.top_k = top_k;
  k.top_p = top_p;
  // 1. the row reducer: chunk maxima (and sums) of every row
  DeviceInfo dev;
  if (device_info(&dev) != SPEC_OK) return SPEC_ERR_CUDA;
  const Plan pl = make_plan(a.B, a.gamma, a.V, sizeof(T), dev.sms, true, kLdg);
  RowStatsParams rp = {};
  rp.target = a.target;
  rp.draft = a.draft;
  rp.temperature = a.temperature;
  rp.partials = reinterpret_cast<float4*>(ws + L.base.partials);
  rp.status = k.status;
  rp.B = a.B;
  rp.gamma = a.gamma;
  rp.V = a.V;
  rp.CE = pl.CE;
  rp.cpr = pl.cpr;
  rp.submax = reinterpret_cast<float*>(ws + L.submax);
  if (launch_pdl(rowstats_kernel<T, kLdg, true>, dim3(pl.grid), dim3(kRowThreads), 0, a.stream, rp) != cudaSuccess)
    return SPEC_ERR_CUDA;
  // 2. K and K' per row (K's superset from the block maxima), 3. the
  // decisions and draws
  k.submax = rp.submax;
  k.cpr = pl.cpr;
  k.CE = pl.CE;
  const int rows = a.B * (2 * a.gamma + 1);
  if (launch_pdl(topk_select_kernel<T>, dim3(rows), dim3(kTkThreads), 0, a.stream, k) != cudaSuccess)
    return SPEC_ERR_CUDA;
  DecideParams& dp = tp.dp;
  dp.target = a.target;
  dp.draft = a.draft;
  dp.draft_tokens = a.draft_tokens;
  dp.temperature = a.temperature;
  dp.u_accept = a.u_accept;
  dp.out_tokens = a.out_tokens;
  dp.out_num = a.out_num;
  dp.out_debug = a.out_debug;
  dp.status = k.status;
  dp.gamma = a.gamma;
  dp.V = a.V;
  tp.u_resample = a.u_resample;
  if (launch_pdl(topkp_tail_kernel<T>, dim3(a.B), dim3(kTkThreads), 0, a.stream, tp) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

// ---------------------------------------------------------------------------
// fused lm_head chain
// ---------------------------------------------------------------------------
// Shape of the lm_head kernel for R hidden rows: the rows are split into
// n_chunks chunks of nc (a multiple of 32, at most 256: the MMA's N), the
// accumulator rotates through n_slots TMEM slots of nc columns, and the two
// TMA rings take what shared memory allows (deeper W ring first).
struct LmPlan {
  int nc, n_chunks, n_slots, w_stages, h_stages;
  uint32_t h_bytes, smem;
};

bool lm_plan(int R, int max_dyn, LmPlan* out) {
  LmPlan p;
  p.n_chunks = (R + kLmMaxChunk - 1) / kLmMaxChunk;
  if (p.n_chunks > 2) return false;  // the kernel issues at most two chunks per K step
  p.nc = (R + 32 * p.n_chunks - 1) / (32 * p.n_chunks) * 32;
  p.n_slots = static_cast<int>(kLmTmemCols) / p.nc;
  if (p.n_slots > kLmMaxSlots) p.n_slots = kLmMaxSlots;
  if (p.n_slots < p.n_chunks) return false;
  p.h_bytes = static_cast<uint32_t>(p.n_chunks * p.nc) * 128u;
  // ring depths in order of preference: the hidden ring waits on L2 round
  // trips every K step, so it keeps its depth before the (prefetched) W ring
  static const int kDepths[][2] = {{5, 6}, {5, 5}, {5, 4}, {4, 4}, {5, 3}, {4, 3}, {3, 3}, {4, 2}, {3, 2}};
  bool fit = false;
  for (const auto& d : kDepths) {
    if (lm_smem_bytes(d[0], d[1], p.h_bytes, p.nc) <= static_cast<uint32_t>(max_dyn)) {
      p.w_stages = d[0];
      p.h_stages = d[1];
      fit = true;
      break;
    }
  }
  if (!fit) return false;
  p.smem = lm_smem_bytes(p.w_stages, p.h_stages, p.h_bytes, p.nc);
  *out = p;
  return true;
}

struct LmLayout {
  Layout base;  // header, draft-row partials, counters
  size_t tpart, logits, rowstat, seq, mass, xsg, total;
  int n_tiles;
};

LmLayout lm_layout(int B, int gamma, int V) {
  LmLayout L;
  L.base = layout(B, gamma, V);
  L.n_tiles = (V + kLmTileV - 1) / kLmTileV;
  const size_t R = static_cast<size_t>(B) * (gamma + 1);
  size_t off = L.base.total;
  L.tpart = off;
  off += align_up(R * L.n_tiles * sizeof(float4), 256);
  L.logits = off;
  off += align_up(static_cast<size_t>(B) * gamma * V * sizeof(float), 256);
  L.rowstat = off;
  off += align_up(static_cast<size_t>(B) * (2 * gamma + 1) * sizeof(RowStat), 256);
  L.seq = off;
  off += align_up(static_cast<size_t>(B) * sizeof(SeqState), 256);
  L.mass = off;
  off += align_up(static_cast<size_t>(B) * L.n_tiles * sizeof(float), 256);
  L.xsg = off;
  off += align_up(static_cast<size_t>(B) * kLmTileV * sizeof(float), 256);
  L.total = off;
  return L;
}

int check_lm_shape(int B, int gamma, int V, int H) {
  if (int e = check_shape(B, gamma, V)) return e;
  if (H < kLmTileK || H > 65536 || (H % kLmTileK) != 0) return SPEC_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * (gamma + 1) > kLmMaxRows) return SPEC_ERR_UNSUPPORTED;
  return SPEC_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::mutex g_encode_mu;

EncodeTiledFn encoder() {
  std::lock_guard<std::mutex> lk(g_encode_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

// 2-D bf16 tensor map over a [rows, H] row-major matrix: boxes of 64 x box_rows
// (128-byte rows, swizzled as the tcgen05 descriptors expect); rows past the
// end read as zero.
bool encode_rows(CUtensorMap* m, const void* base, int rows, int H, int box_rows) {
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kLmTileK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct LmArgs {
  const void* hidden;
  const void* W;
  const void* draft;
  const int32_t* draft_tokens;
  const float* temperature;
  const float* u_accept;
  const float* u_resample;
  int B, gamma, V, H;
  int32_t* out_tokens;
  int32_t* out_num;
  float* out_debug;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  bool gemm_only;  // launch only the lm_head kernel (timing / profiling)
};

int run_lm_chain(const LmArgs& a) {
  const LmLayout L = lm_layout(a.B, a.gamma, a.V);
  if (a.ws_bytes < L.total) return SPEC_ERR_WORKSPACE;
  DeviceInfo dev;
  if (device_info(&dev) != SPEC_OK) return SPEC_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  int* status = reinterpret_cast<int*>(ws + L.base.header);
  const int R = a.B * (a.gamma + 1);

  // 1. draft rows: chunk partials (the row reducer's items, target rows
  // skipped), computed by the GEMM kernel's row warps
  const Plan pl = make_plan_rows(a.B * a.gamma, a.V, sizeof(__nv_bfloat16), dev.sms, kLdg);
  RowStatsParams rp = {};
  rp.target = nullptr;
  rp.draft = a.draft;
  rp.temperature = a.temperature;
  rp.partials = reinterpret_cast<float4*>(ws + L.base.partials);
  rp.status = status;
  rp.B = a.B;
  rp.gamma = a.gamma;
  rp.V = a.V;
  rp.CE = pl.CE;
  rp.cpr = pl.cpr;
  rp.draft_only = 1;

  // 2. target rows: the lm_head GEMM with its statistics epilogue (same kernel)
  LmPlan plan;
  if (!lm_plan(R, dev.lm_max_dyn, &plan)) return SPEC_ERR_UNSUPPORTED;
  LmParams lp;
  std::memset(&lp, 0, sizeof(lp));
  if (!encode_rows(&lp.tmW, a.W, a.V, a.H, kLmTileV) || !encode_rows(&lp.tmH, a.hidden, R, a.H, plan.nc))
    return SPEC_ERR_CUDA;
  lp.R = R;
  lp.V = a.V;
  lp.H = a.H;
  lp.n_tiles = L.n_tiles;
  lp.gamma = a.gamma;
  lp.nc = plan.nc;
  lp.n_chunks = plan.n_chunks;
  lp.n_slots = plan.n_slots;
  lp.w_stages = plan.w_stages;
  lp.h_stages = plan.h_stages;
  lp.h_bytes = plan.h_bytes;
  lp.temperature = a.temperature;
  lp.partials = reinterpret_cast<float4*>(ws + L.tpart);
  lp.logits = reinterpret_cast<float*>(ws + L.logits);
  lp.status = status;
  // the draft rows' statistics come from the GEMM kernel's row warps (none
  // when only the GEMM is timed)
  lp.rows = rp;
  if (a.gemm_only) lp.rows.draft = nullptr;
  const int lm_grid = L.n_tiles < dev.sms ? L.n_tiles : dev.sms;
  // first kernel of the call: plain stream order (the previous call's last
  // kernel still reads this workspace)
  if (plan.n_chunks == 1)
    lmhead_kernel<1><<<lm_grid, kLmThreads, plan.smem, a.stream>>>(lp);
  else
    lmhead_kernel<2><<<lm_grid, kLmThreads, plan.smem, a.stream>>>(lp);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (a.gemm_only) return SPEC_OK;

  // 3. decision, 4. residual / bonus masses and the draw
  LmTailParams tp = {};
  tp.hidden = static_cast<const __nv_bfloat16*>(a.hidden);
  tp.W = static_cast<const __nv_bfloat16*>(a.W);
  tp.draft = static_cast<const __nv_bfloat16*>(a.draft);
  tp.logits = lp.logits;
  tp.tpart = lp.partials;
  tp.dpart = rp.partials;
  tp.rowstat = reinterpret_cast<RowStat*>(ws + L.rowstat);
  tp.seq = reinterpret_cast<SeqState*>(ws + L.seq);
  tp.mass = reinterpret_cast<float*>(ws + L.mass);
  tp.xsg = reinterpret_cast<float*>(ws + L.xsg);
  tp.tail_done = reinterpret_cast<int*>(ws + L.base.tail_done);
  tp.u_resample = a.u_resample;
  tp.B = a.B;
  tp.gamma = a.gamma;
  tp.V = a.V;
  tp.H = a.H;
  tp.n_tiles = L.n_tiles;
  tp.cpr_d = pl.cpr;
  DecideParams& dp = tp.dp;
  dp.target = nullptr;
  dp.draft = a.draft;
  dp.draft_tokens = a.draft_tokens;
  dp.temperature = a.temperature;
  dp.u_accept = a.u_accept;
  dp.out_tokens = a.out_tokens;
  dp.out_num = a.out_num;
  dp.out_debug = a.out_debug;
  dp.status = status;
  dp.gamma = a.gamma;
  dp.V = a.V;
  if (launch_pdl(lm_decide_kernel, dim3(a.B), dim3(kLmTailThreads), 0, a.stream, tp) != cudaSuccess)
    return SPEC_ERR_CUDA;
  // parts per sequence: three CTAs per SM (76 registers x 256 threads) over the
  // batch, rounded down so every CTA is resident in one wave, >= 8 tiles each
  // (rounding up left a second wave of 56 CTAs at B=64: 1.4 us per round)
  int parts = (3 * dev.sms) / a.B;
  if (parts > L.n_tiles / 8) parts = L.n_tiles / 8;
  if (parts > 64) parts = 64;
  if (parts < 1) parts = 1;
  if (launch_pdl(lm_tail_kernel, dim3(parts, a.B), dim3(kLmTailThreads), 0, a.stream, tp) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// centroid-masked draft head and verification against its sparse rows
// ---------------------------------------------------------------------------
struct HeadLayout {
  size_t header, scores, sel, pos, total;
};

// Shape of the cluster-score GEMM for R hidden rows: row chunks of N (a
// multiple of 16, at most 256), and at most sc_max_split(R, n_clusters) K
// parts: split K only while there are few tiles (a few dozen CTAs at most
// otherwise), which also bounds the partial-score workspace.
int sc_rows_n(int R) { return R >= kScMaxN ? kScMaxN : ((R + 15) / 16) * 16; }
int sc_max_split(int R, int n_clusters) {
  const long long tiles = (n_clusters + kScTileC - 1) / kScTileC;
  const long long chunks = (R + sc_rows_n(R) - 1) / sc_rows_n(R);
  return tiles * chunks <= 64 ? kScMaxSplit : 1;
}

HeadLayout head_layout(int R, int n_clusters, int top_k) {
  HeadLayout L;
  size_t off = 0;
  L.header = off;
  off += align_up(sizeof(WsHeader), 256);
  L.scores = off;  // the K parts' partial scores
  off += align_up(static_cast<size_t>(sc_max_split(R, n_clusters)) * R * n_clusters * sizeof(float), 256);
  L.sel = off;
  off += align_up(static_cast<size_t>(R) * top_k * sizeof(int32_t), 256);
  L.pos = off;
  off += align_up(static_cast<size_t>(R) * (top_k + 1) * sizeof(int32_t), 256);
  L.total = off;
  return L;
}

int pow2_at_least(int n) {
  int p2 = 1;
  while (p2 < n) p2 <<= 1;
  return p2;
}

struct SparseLayout {
  Layout base;
  size_t cand_lo, total;
};

SparseLayout sparse_layout(int B, int gamma, int V) {
  SparseLayout L;
  L.base = layout(B, gamma, V);
  const size_t cpr = (static_cast<size_t>(V) + kMinChunk - 1) / kMinChunk;
  L.cand_lo = L.base.total;
  L.total = L.cand_lo + align_up(static_cast<size_t>(B) * (cpr + 1) * sizeof(int32_t), 256);
  return L;
}

struct SparseArgs {
  const int32_t* cand_tok;
  const float* cand_logit;
  const int32_t* cand_count;
  int stride;
};

template <typename T>
int run_sparse(const Common& a, const SparseArgs& c) {
  const SparseLayout L = sparse_layout(a.B, a.gamma, a.V);
  if (a.ws_bytes < L.total) return SPEC_ERR_WORKSPACE;
  DeviceInfo dev;
  if (device_info(&dev) != SPEC_OK) return SPEC_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  int* status = reinterpret_cast<int*>(ws + L.base.header);
  const Plan pl = make_plan(a.B, a.gamma, a.V, sizeof(T), dev.sms, true, kLdg);
  RowStatsParams rp = {};
  rp.target = a.target;
  rp.draft = nullptr;  // the draft rows are sparse: never streamed
  rp.temperature = a.temperature;
  rp.partials = reinterpret_cast<float4*>(ws + L.base.partials);
  rp.status = status;
  rp.B = a.B;
  rp.gamma = a.gamma;
  rp.V = a.V;
  rp.CE = pl.CE;
  rp.cpr = pl.cpr;
  if (launch_pdl(rowstats_kernel<T, kLdg>, dim3(pl.grid), dim3(kRowThreads), 0, a.stream, rp) != cudaSuccess)
    return SPEC_ERR_CUDA;
  SparseParams sp = {};
  sp.target = a.target;
  sp.cand_tok = c.cand_tok;
  sp.cand_logit = c.cand_logit;
  sp.cand_count = c.cand_count;
  sp.u_resample = a.u_resample;
  sp.partials = rp.partials;
  sp.mass = reinterpret_cast<float*>(ws + L.base.mass);
  sp.cand_lo = reinterpret_cast<int32_t*>(ws + L.cand_lo);
  sp.tail_done = reinterpret_cast<int*>(ws + L.base.tail_done);
  sp.B = a.B;
  sp.gamma = a.gamma;
  sp.V = a.V;
  sp.CE = pl.CE;
  sp.cpr = pl.cpr;
  sp.stride = c.stride;
  DecideParams& dp = sp.dp;
  dp.target = a.target;
  dp.draft = nullptr;
  dp.draft_tokens = a.draft_tokens;
  dp.temperature = a.temperature;
  dp.u_accept = a.u_accept;
  dp.out_tokens = a.out_tokens;
  dp.out_num = a.out_num;
  dp.out_debug = a.out_debug;
  dp.status = status;
  dp.gamma = a.gamma;
  dp.V = a.V;
  // one tail CTA per SM over the batch (at most 16 per sequence); two per SM
  // (64 registers, 9 parts for B=32) measured the same
  int parts = dev.sms / a.B;
  if (parts > 16) parts = 16;
  if (parts > pl.cpr) parts = pl.cpr;
  if (parts < 1) parts = 1;
  if (launch_pdl(sparse_tail_kernel<T>, dim3(parts, a.B), dim3(kSparseThreads), 0, a.stream, sp) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

extern "C" {

int spec_verify_version(void) { return 200; }

const char* spec_verify_error_string(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported dtype or shape";
    case SPEC_ERR_ALIGNMENT: return "logit pointer not 16-byte aligned";
    case SPEC_ERR_WORKSPACE: return "workspace null, misaligned or too small";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    case SPEC_ERR_TIMEOUT: return "device wait timed out";
    case SPEC_ERR_DEVICE_INPUT: return "draft token outside [0, V)";
    case SPEC_ERR_STATE: return "inconsistent round bookkeeping (kv_len != seq_len - 1 or accepted > gamma)";
    case SPEC_ERR_DEVICE_BOUNDS: return "device index outside its extent (bounds-checked build)";
    default: return "unknown error";
  }
}

int spec_verify_workspace_bytes(int B, int gamma, int V, int H, size_t* bytes) {
  if (bytes == nullptr) return SPEC_ERR_INVALID_ARG;
  if (H == 0) {
    if (check_shape(B, gamma, V) != SPEC_OK) return SPEC_ERR_INVALID_ARG;
    *bytes = layout(B, gamma, V).total;
    return SPEC_OK;
  }
  if (int e = check_lm_shape(B, gamma, V, H)) return e;
  *bytes = lm_layout(B, gamma, V).total;
  return SPEC_OK;
}

int spec_verify_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr) return SPEC_ERR_WORKSPACE;
  if (cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

int spec_verify_greedy(const void* target_logits, spec_dtype dt, const int32_t* draft_tokens, int B,
                       int gamma, int V, int32_t* out_tokens, int32_t* out_num_accepted, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (target_logits == nullptr || draft_tokens == nullptr || out_tokens == nullptr ||
      out_num_accepted == nullptr)
    return SPEC_ERR_INVALID_ARG;
  if (int e = check_shape(B, gamma, V)) return e;
  if (dt != SPEC_F32 && dt != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(target_logits)) return SPEC_ERR_ALIGNMENT;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return SPEC_ERR_WORKSPACE;
  Common a = {};
  a.target = target_logits;
  a.dt = dt;
  a.draft_tokens = draft_tokens;
  a.B = B;
  a.gamma = gamma;
  a.V = V;
  a.out_tokens = out_tokens;
  a.out_num = out_num_accepted;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  return dispatch(a, false);
}

int spec_verify_greedy_multi(const void* target_logits, spec_dtype dt, const int32_t* draft_tokens, int B,
                             int n_cand, int gamma, int V, int32_t* out_tokens, int32_t* out_num_accepted,
                             int32_t* out_choice, void* workspace, size_t workspace_bytes, void* stream) {
  if (target_logits == nullptr || draft_tokens == nullptr || out_tokens == nullptr ||
      out_num_accepted == nullptr)
    return SPEC_ERR_INVALID_ARG;
  if (n_cand < 1 || B < 1 || static_cast<long long>(B) * n_cand > 65535) return SPEC_ERR_INVALID_ARG;
  const int BN = B * n_cand;
  if (int e = check_shape(BN, gamma, V)) return e;
  if (dt != SPEC_F32 && dt != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(target_logits)) return SPEC_ERR_ALIGNMENT;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return SPEC_ERR_WORKSPACE;
  const Layout L = layout(BN, gamma, V);
  if (workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  // every candidate is verified greedily as a sequence of its own (rows
  // b*n_cand + c), into the workspace; then one warp per sequence keeps the
  // best candidate
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* cand_tokens = reinterpret_cast<int32_t*>(ws + L.cand);
  int32_t* cand_num = cand_tokens + static_cast<size_t>(BN) * (gamma + 1);
  Common a = {};
  a.target = target_logits;
  a.dt = dt;
  a.draft_tokens = draft_tokens;
  a.B = BN;
  a.gamma = gamma;
  a.V = V;
  a.out_tokens = cand_tokens;
  a.out_num = cand_num;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  if (int e = dispatch(a, false)) return e;
  if (launch_pdl(select_candidate_kernel, dim3(B), dim3(32), 0, a.stream, cand_tokens,
                 static_cast<const int32_t*>(cand_num), n_cand, gamma, out_tokens, out_num_accepted,
                 out_choice) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

static int sample_entry(bool reduce_only, const void* target_logits, const void* draft_logits, spec_dtype dt,
                       const int32_t* draft_tokens, const float* temperature, const float* u_accept,
                       const float* u_resample, int B, int gamma, int V, int32_t* out_tokens,
                       int32_t* out_num_accepted, float* out_debug, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (target_logits == nullptr || draft_logits == nullptr || draft_tokens == nullptr ||
      temperature == nullptr || u_accept == nullptr || u_resample == nullptr || out_tokens == nullptr ||
      out_num_accepted == nullptr)
    return SPEC_ERR_INVALID_ARG;
  if (int e = check_shape(B, gamma, V)) return e;
  if (dt != SPEC_F32 && dt != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(target_logits) || !aligned16(draft_logits)) return SPEC_ERR_ALIGNMENT;
  if (out_debug != nullptr && !aligned16(out_debug)) return SPEC_ERR_ALIGNMENT;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return SPEC_ERR_WORKSPACE;
  Common a = {};
  a.target = target_logits;
  a.draft = draft_logits;
  a.dt = dt;
  a.draft_tokens = draft_tokens;
  a.temperature = temperature;
  a.u_accept = u_accept;
  a.u_resample = u_resample;
  a.B = B;
  a.gamma = gamma;
  a.V = V;
  a.out_tokens = out_tokens;
  a.out_num = out_num_accepted;
  a.out_debug = out_debug;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  a.reduce_only = reduce_only;
  return dispatch(a, true);
}

int spec_verify_sample(const void* target_logits, const void* draft_logits, spec_dtype dt,
                       const int32_t* draft_tokens, const float* temperature, const float* u_accept,
                       const float* u_resample, int B, int gamma, int V, int32_t* out_tokens,
                       int32_t* out_num_accepted, float* out_debug, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return sample_entry(false, target_logits, draft_logits, dt, draft_tokens, temperature, u_accept,
                      u_resample, B, gamma, V, out_tokens, out_num_accepted, out_debug, workspace,
                      workspace_bytes, stream);
}

int spec_verify_sample_reduce_only(const void* target_logits, const void* draft_logits, spec_dtype dt,
                                   const int32_t* draft_tokens, const float* temperature,
                                   const float* u_accept, const float* u_resample, int B, int gamma,
                                   int V, int32_t* out_tokens, int32_t* out_num_accepted,
                                   float* out_debug, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  return sample_entry(true, target_logits, draft_logits, dt, draft_tokens, temperature, u_accept,
                      u_resample, B, gamma, V, out_tokens, out_num_accepted, out_debug, workspace,
                      workspace_bytes, stream);
}

static int lmhead_entry(bool gemm_only, const void* hidden, const void* W, const void* draft_logits,
                        const int32_t* draft_tokens, const float* temperature, const float* u_accept,
                        const float* u_resample, int B, int gamma, int V, int H, int32_t* out_tokens,
                        int32_t* out_num_accepted, float* out_debug, void* workspace, size_t workspace_bytes,
                        void* stream) {
  if (hidden == nullptr || W == nullptr || draft_logits == nullptr || draft_tokens == nullptr ||
      temperature == nullptr || u_accept == nullptr || u_resample == nullptr || out_tokens == nullptr ||
      out_num_accepted == nullptr)
    return SPEC_ERR_INVALID_ARG;
  if (int e = check_lm_shape(B, gamma, V, H)) return e;
  if (!aligned16(hidden) || !aligned16(W) || !aligned16(draft_logits)) return SPEC_ERR_ALIGNMENT;
  if (out_debug != nullptr && !aligned16(out_debug)) return SPEC_ERR_ALIGNMENT;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return SPEC_ERR_WORKSPACE;
  LmArgs a = {};
  a.hidden = hidden;
  a.W = W;
  a.draft = draft_logits;
  a.draft_tokens = draft_tokens;
  a.temperature = temperature;
  a.u_accept = u_accept;
  a.u_resample = u_resample;
  a.B = B;
  a.gamma = gamma;
  a.V = V;
  a.H = H;
  a.out_tokens = out_tokens;
  a.out_num = out_num_accepted;
  a.out_debug = out_debug;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  a.gemm_only = gemm_only;
  return run_lm_chain(a);
}

int spec_verify_lmhead_sample(const void* hidden, const void* W, const void* draft_logits,
                              const int32_t* draft_tokens, const float* temperature, const float* u_accept,
                              const float* u_resample, int B, int gamma, int V, int H, int32_t* out_tokens,
                              int32_t* out_num_accepted, float* out_debug, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return lmhead_entry(false, hidden, W, draft_logits, draft_tokens, temperature, u_accept, u_resample, B, gamma,
                      V, H, out_tokens, out_num_accepted, out_debug, workspace, workspace_bytes, stream);
}

int spec_verify_lmhead_gemm_only(const void* hidden, const void* W, const void* draft_logits,
                                 const int32_t* draft_tokens, const float* temperature, const float* u_accept,
                                 const float* u_resample, int B, int gamma, int V, int H, int32_t* out_tokens,
                                 int32_t* out_num_accepted, float* out_debug, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return lmhead_entry(true, hidden, W, draft_logits, draft_tokens, temperature, u_accept, u_resample, B, gamma,
                      V, H, out_tokens, out_num_accepted, out_debug, workspace, workspace_bytes, stream);
}

int spec_verify_topkp_workspace_bytes(int B, int gamma, int V, size_t* bytes) {
  if (bytes == nullptr || check_shape(B, gamma, V) != SPEC_OK) return SPEC_ERR_INVALID_ARG;
  *bytes = tk_layout(B, gamma, V).total;
  return SPEC_OK;
}

int spec_verify_sample_topkp(const void* target_logits, const void* draft_logits, spec_dtype dt,
                             const int32_t* draft_tokens, const float* temperature, const float* u_accept,
                             const float* u_resample, int B, int gamma, int V, int top_k, float top_p,
                             int32_t* out_tokens, int32_t* out_num_accepted, float* out_debug, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (target_logits == nullptr || draft_logits == nullptr || draft_tokens == nullptr ||
      temperature == nullptr || u_accept == nullptr || u_resample == nullptr || out_tokens == nullptr ||
      out_num_accepted == nullptr)
    return SPEC_ERR_INVALID_ARG;
  if (int e = check_shape(B, gamma, V)) return e;
  if (top_k < 1 || top_k > kTkMaxK || !(top_p > 0.f && top_p <= 1.f)) return SPEC_ERR_INVALID_ARG;
  if (dt != SPEC_F32 && dt != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(target_logits) || !aligned16(draft_logits)) return SPEC_ERR_ALIGNMENT;
  if (out_debug != nullptr && !aligned16(out_debug)) return SPEC_ERR_ALIGNMENT;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return SPEC_ERR_WORKSPACE;
  Common a = {};
  a.target = target_logits;
  a.draft = draft_logits;
  a.dt = dt;
  a.draft_tokens = draft_tokens;
  a.temperature = temperature;
  a.u_accept = u_accept;
  a.u_resample = u_resample;
  a.B = B;
  a.gamma = gamma;
  a.V = V;
  a.out_tokens = out_tokens;
  a.out_num = out_num_accepted;
  a.out_debug = out_debug;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  return dt == SPEC_F32 ? run_topkp<float>(a, top_k, top_p) : run_topkp<__nv_bfloat16>(a, top_k, top_p);
}

int spec_centroid_head_workspace_bytes(int R, int n_clusters, int top_k, size_t* bytes) {
  if (bytes == nullptr || R < 1 || R > 65535 || n_clusters < 1 || n_clusters > kHeadMaxClusters || top_k < 1 ||
      top_k > n_clusters || top_k > kHeadMaxTopK)
    return SPEC_ERR_INVALID_ARG;
  *bytes = head_layout(R, n_clusters, top_k).total;
  return SPEC_OK;
}

int spec_centroid_head(const void* hidden, const void* centroids, const void* W_ord, const int32_t* cluster_off,
                       const int32_t* ord2tok, int R, int H, int V, int n_clusters, int top_k, int max_cand,
                       int32_t* out_tok, float* out_logit, int32_t* out_count, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (hidden == nullptr || centroids == nullptr || W_ord == nullptr || cluster_off == nullptr ||
      ord2tok == nullptr || out_tok == nullptr || out_logit == nullptr || out_count == nullptr)
    return SPEC_ERR_INVALID_ARG;
  if (R < 1 || R > 65535 || H < 256 || H > 256 * kHeadMaxVecs || (H % 256) != 0 || V < 1 ||
      V > SPEC_MAX_VOCAB || n_clusters < 1 || n_clusters > kHeadMaxClusters || top_k < 1 || top_k > n_clusters ||
      top_k > kHeadMaxTopK || max_cand < 1 || max_cand > kHeadMaxCand)
    return SPEC_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(centroids) || !aligned16(W_ord)) return SPEC_ERR_ALIGNMENT;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPEC_ERR_WORKSPACE;
  const HeadLayout L = head_layout(R, n_clusters, top_k);
  if (workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  DeviceInfo dev;
  if (device_info(&dev) != SPEC_OK) return SPEC_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  HeadParams hp;
  hp.hidden = static_cast<const __nv_bfloat16*>(hidden);
  hp.centroids = static_cast<const __nv_bfloat16*>(centroids);
  hp.W_ord = static_cast<const __nv_bfloat16*>(W_ord);
  hp.cluster_off = cluster_off;
  hp.ord2tok = ord2tok;
  hp.scores = reinterpret_cast<float*>(ws + L.scores);
  hp.sel = reinterpret_cast<int32_t*>(ws + L.sel);
  hp.pos = reinterpret_cast<int32_t*>(ws + L.pos);
  hp.out_tok = out_tok;
  hp.out_logit = out_logit;
  hp.out_count = out_count;
  hp.status = reinterpret_cast<int*>(ws + L.header);
  hp.R = R;
  hp.H = H;
  hp.V = V;
  hp.n_clusters = n_clusters;
  hp.top_k = top_k;
  hp.max_cand = max_cand;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the score GEMM (more than kHeadScoreTcRows rows): 128-centroid tiles x
  // row chunks, K split so that the grid has about two CTAs per SM
  const bool sc_tc = R > kHeadScoreTcRows;
  ScoreParams sp;
  std::memset(&sp, 0, sizeof(sp));
  sp.N = sc_rows_n(R);
  if (sc_tc && (!encode_rows(&sp.tmC, centroids, n_clusters, H, kScTileC) ||
                !encode_rows(&sp.tmH, hidden, R, H, sp.N)))
    return SPEC_ERR_CUDA;
  const int tiles = (n_clusters + kScTileC - 1) / kScTileC, chunks = (R + sp.N - 1) / sp.N;
  const int ksteps = H / kScK;
  int ksplit = (2 * dev.sms + tiles * chunks - 1) / (tiles * chunks);
  const int max_split = sc_max_split(R, n_clusters);
  if (ksplit > max_split) ksplit = max_split;
  if (ksplit > ksteps) ksplit = ksteps;
  if (ksplit < 1) ksplit = 1;
  sp.kper = (ksteps + ksplit - 1) / ksplit;
  sp.ksplit = (ksteps + sp.kper - 1) / sp.kper;  // no empty part
  sp.scores = hp.scores;
  sp.status = hp.status;
  sp.R = R;
  sp.H = H;
  sp.n_clusters = n_clusters;
  hp.ksplit = sc_tc ? sp.ksplit : 1;
  const size_t sc_smem = static_cast<size_t>(kScStages) * sc_stage_bytes(sp.N) + 1024;
  const size_t sort1 = static_cast<size_t>(n_clusters) * sizeof(uint32_t);
  const size_t sort2 = (V <= kHeadBitmapV) ? kHeadSortSmemBitmap
                                           : static_cast<size_t>(pow2_at_least(max_cand)) * sizeof(unsigned long long);
  const cudaError_t e_sc =
      sc_tc ? launch_pdl(cluster_score_tc_kernel, dim3(tiles * sp.ksplit, chunks), dim3(kScThreads), sc_smem, st, sp)
            : launch_pdl(cluster_score_cc_kernel,
                         dim3((n_clusters + kHeadWarps - 1) / kHeadWarps, (R + kHeadRowBlock - 1) / kHeadRowBlock),
                         dim3(kHeadThreads), 0, st, hp);
  if (e_sc != cudaSuccess ||
      launch_pdl(cluster_topk_kernel, dim3(R), dim3(kHeadThreads), sort1, st, hp) != cudaSuccess ||
      launch_pdl(cand_logit_kernel, dim3(top_k, R), dim3(kHeadThreads), 0, st, hp) != cudaSuccess ||
      launch_pdl(cand_sort_kernel, dim3(R), dim3(kHeadThreads), sort2, st, hp) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

int spec_verify_sparse_workspace_bytes(int B, int gamma, int V, size_t* bytes) {
  if (bytes == nullptr || check_shape(B, gamma, V) != SPEC_OK) return SPEC_ERR_INVALID_ARG;
  *bytes = sparse_layout(B, gamma, V).total;
  return SPEC_OK;
}

int spec_verify_sample_sparse(const void* target_logits, spec_dtype dt, const int32_t* cand_tok,
                              const float* cand_logit, const int32_t* cand_count, int cand_stride,
                              const int32_t* draft_tokens, const float* temperature, const float* u_accept,
                              const float* u_resample, int B, int gamma, int V, int32_t* out_tokens,
                              int32_t* out_num_accepted, float* out_debug, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (target_logits == nullptr || cand_tok == nullptr || cand_logit == nullptr || cand_count == nullptr ||
      draft_tokens == nullptr || temperature == nullptr || u_accept == nullptr || u_resample == nullptr ||
      out_tokens == nullptr || out_num_accepted == nullptr)
    return SPEC_ERR_INVALID_ARG;
  if (int e = check_shape(B, gamma, V)) return e;
  if (cand_stride < 1) return SPEC_ERR_INVALID_ARG;
  if (dt != SPEC_F32 && dt != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(target_logits)) return SPEC_ERR_ALIGNMENT;
  if (out_debug != nullptr && !aligned16(out_debug)) return SPEC_ERR_ALIGNMENT;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPEC_ERR_WORKSPACE;
  Common a = {};
  a.target = target_logits;
  a.dt = dt;
  a.draft_tokens = draft_tokens;
  a.temperature = temperature;
  a.u_accept = u_accept;
  a.u_resample = u_resample;
  a.B = B;
  a.gamma = gamma;
  a.V = V;
  a.out_tokens = out_tokens;
  a.out_num = out_num_accepted;
  a.out_debug = out_debug;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  const SparseArgs c{cand_tok, cand_logit, cand_count, cand_stride};
  return dt == SPEC_F32 ? run_sparse<float>(a, c) : run_sparse<__nv_bfloat16>(a, c);
}

int spec_verify_status(void* workspace, void* stream) {
  if (workspace == nullptr) return SPEC_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SPEC_ERR_CUDA;
  if (st != 0 && cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return SPEC_ERR_CUDA;
  if (st & kStatusTimeout) return SPEC_ERR_TIMEOUT;
  if (st & kStatusBadToken) return SPEC_ERR_DEVICE_INPUT;
  if (st & (kStatusTopkOverflow | kStatusLimit)) return SPEC_ERR_UNSUPPORTED;
  if (st & kStatusBounds) return SPEC_ERR_DEVICE_BOUNDS;
  return SPEC_OK;
}

int spec_verify_selftest_timeout(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return SPEC_ERR_WORKSPACE;
  if (workspace_bytes < layout(1, 1, 8).total) return SPEC_ERR_WORKSPACE;
  // one tiny launch whose only wait can never be satisfied (~1 ms limit)
  Common a = {};
  a.B = 1;
  a.gamma = 1;
  a.V = 8;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  a.debug = 1;
  a.target = workspace;  // never read in this mode
  return run_chain<float>(a, false);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: a plugin or custom op inside an
// inference engine that owns every byte of device memory through its own
// pool, or a latency-critical decode loop where an allocation could
// synchronise the device and stall the other streams.  For them
// spec_verify_sample_noalloc keeps its scratch in the array below, a fixed
// 16 MiB in every GPU that loads this library, held until the process exits.
// The caller still passes all inputs and outputs.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
struct NoAllocDevice {
  void* ptr = nullptr;  // device address of g_noalloc_scratch on this device
  bool ready = false;
};
NoAllocDevice g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

// Once per device, with that device current: look up the array's device
// address (its name is only a stand-in in host code).  Nothing is written
// here: each call clears, on the caller's stream, what must start at zero.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SPEC_ERR_CUDA;
    d.ptr = p;
    d.ready = true;
  }
  *out = d.ptr;
  return SPEC_OK;
}
}  // namespace

extern "C" int spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                                          spec_dtype dt, const int32_t* draft_tokens,
                                          const float* temperature, const float* u_accept,
                                          const float* u_resample, int B, int gamma, int V,
                                          int32_t* out_tokens, int32_t* out_num_accepted,
                                          float* out_debug, void* stream) {
  // the same checks as spec_verify_sample, before any CUDA call
  if (target_logits == nullptr || draft_logits == nullptr || draft_tokens == nullptr ||
      temperature == nullptr || u_accept == nullptr || u_resample == nullptr || out_tokens == nullptr ||
      out_num_accepted == nullptr)
    return SPEC_ERR_INVALID_ARG;
  if (int e = check_shape(B, gamma, V)) return e;
  if (dt != SPEC_F32 && dt != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(target_logits) || !aligned16(draft_logits)) return SPEC_ERR_ALIGNMENT;
  if (out_debug != nullptr && !aligned16(out_debug)) return SPEC_ERR_ALIGNMENT;
  const Layout L = layout(B, gamma, V);
  if (L.total > kNoAllocScratchBytes) return SPEC_ERR_WORKSPACE;  // beyond the built-in scratch
  void* scratch = nullptr;
  if (int e = noalloc_scratch(&scratch)) return e;
  // the header (status word) and the per-sequence counters must start at
  // zero; everything else in the scratch is written before it is read.  Both
  // clears go on the caller's stream, ahead of the kernels.
  unsigned char* sc = static_cast<unsigned char*>(scratch);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(sc + L.header, 0, L.partials - L.header, st) != cudaSuccess ||
      cudaMemsetAsync(sc + L.tail_done, 0, L.total - L.tail_done, st) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return spec_verify_sample(target_logits, draft_logits, dt, draft_tokens, temperature, u_accept,
                            u_resample, B, gamma, V, out_tokens, out_num_accepted, out_debug, scratch,
                            kNoAllocScratchBytes, stream);
}
