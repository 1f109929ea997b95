// Host side of the FLARE++ mixer forward: argument validation, the workspace
// plan and cache, the split heuristic and the kernel launches behind the C
// ABI of include/flarepp.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdio>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "flarepp.h"
#include "common.cuh"
#include "launch.h"
#include "simt.cuh"

namespace flarepp {
namespace {

std::atomic<int> g_forced_splits{0};
std::atomic<int> g_fail_wait{0};  // test hook: see flarepp_test_fail_wait
thread_local char g_last_error[256] = "no error";
cudaEvent_t* g_stage_events = nullptr;

// Records which CUDA call failed (for flarepp_last_error) and passes the result on.
bool cuda_ok(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return true;
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", what, cudaGetErrorName(e),
           cudaGetErrorString(e));
  return false;
}

bool stage_event(int i, cudaStream_t stream) {
  if (g_stage_events == nullptr) return true;
  return cuda_ok(cudaEventRecord(g_stage_events[i], stream), "cudaEventRecord(stage event)");
}

struct Problem {
  int variant = kVariantFlarePP;
  const void* K;
  const void* V;
  const void* Ks;
  const void* Vs;
  const void* Qseed;
  const void* Qf;
  const float* gate;
  const void* Q;
  int B, H, N, M, D;
  flarepp_dtype_t dtype;
  void* out;
  float* dbg_qd;
  float* dbg_q;
  float* dbg_z;
  float* dbg_l;
};

size_t elem_size(flarepp_dtype_t t) { return t == FLAREPP_BF16 ? 2 : 4; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

flarepp_status_t check_sizes(int B, int H, int N, int M, int D, flarepp_dtype_t dtype) {
  if (B <= 0 || H <= 0 || N <= 0 || M <= 0 || D <= 0) return FLAREPP_ERR_INVALID_ARG;
  if (dtype != FLAREPP_BF16 && dtype != FLAREPP_FP32) return FLAREPP_ERR_UNSUPPORTED;
  if (D != 16 && D != 32) return FLAREPP_ERR_UNSUPPORTED;
  if (M > 512) return FLAREPP_ERR_UNSUPPORTED;
  if (dtype == FLAREPP_BF16 && M % 16 != 0) return FLAREPP_ERR_UNSUPPORTED;
  const long long tokens = (long long)B * H * N * D;
  if (tokens >= (1LL << 31)) return FLAREPP_ERR_UNSUPPORTED;
  if ((long long)B * H > 65535) return FLAREPP_ERR_UNSUPPORTED;
  return FLAREPP_OK;
}

// The inputs a variant reads: every one must be given, and the others must
// be null (a pointer the call would ignore is more likely a mistake).
struct Needs {
  bool Ks, Vs, Qseed, Qf, gate, Q;
};
Needs needs_of(int variant) {
  switch (variant) {
    case kVariantFlarePP: return {true, false, true, true, true, false};
    case kVariantUnshared: return {true, true, true, true, true, false};
    case kVariantSimplified: return {true, true, true, false, false, false};
    default: return {false, false, false, false, false, true};  // FLARE
  }
}

flarepp_status_t validate(const Problem& p) {
  flarepp_status_t st = check_sizes(p.B, p.H, p.N, p.M, p.D, p.dtype);
  if (st != FLAREPP_OK) return st;
  if (p.variant < kVariantFlarePP || p.variant > kVariantFlare) return FLAREPP_ERR_INVALID_ARG;
  const Needs n = needs_of(p.variant);
  const std::pair<const void*, bool> opt[] = {{p.Ks, n.Ks}, {p.Vs, n.Vs}, {p.Qseed, n.Qseed},
                                              {p.Qf, n.Qf}, {p.gate, n.gate}, {p.Q, n.Q}};
  if (p.K == nullptr || p.V == nullptr || p.out == nullptr) return FLAREPP_ERR_INVALID_ARG;
  for (const auto& o : opt)
    if ((o.first != nullptr) != o.second) return FLAREPP_ERR_INVALID_ARG;
  const void* all[] = {p.K, p.V, p.Ks, p.Vs, p.Qseed, p.Qf, p.gate, p.Q, p.out,
                       p.dbg_qd, p.dbg_q, p.dbg_z, p.dbg_l};
  for (const void* ptr : all)
    if (ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return FLAREPP_ERR_ALIGNMENT;
  const size_t es = elem_size(p.dtype);
  const size_t tok = (size_t)p.B * p.H * p.N * p.D * es;
  const size_t lat = (size_t)p.H * p.M * p.D * es;
  const std::pair<const void*, size_t> inputs[] = {
      {p.K, tok},     {p.V, tok},  {p.Ks, tok}, {p.Vs, tok}, {p.Qseed, lat},
      {p.Qf, lat},    {p.Q, lat},  {p.gate, (size_t)p.H * 4}};
  for (const auto& in : inputs)
    if (in.first != nullptr && overlaps(p.out, tok, in.first, in.second)) return FLAREPP_ERR_INVALID_ARG;
  return FLAREPP_OK;
}

// Workspace layout. Both split-N passes run one after the other on the
// stream, so they share the partial-result buffers; each has its own set of
// arrival counters, which the last CTA of every group resets to zero.
struct Plan {
  int BH = 0, tiles = 0, splits = 0, split_len = 0;
  TcPlan tc{};  // bf16 tensor-core path
  size_t off_pz = 0, off_pl = 0, off_cnt = 0, off_q = 0, off_z = 0, total = 0;
};

int device_sm_count() {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev] = sms;
  return sms;
}

// fp32 path: enough (split, tile, head) CTAs to give every SM about two, each
// split a whole number of staged tiles. bf16 path: tc_plan (tc.cu).
Plan make_plan(int B, int H, int N, int M, int D, flarepp_dtype_t dtype, int sms) {
  Plan pl;
  pl.BH = B * H;
  size_t rows = 0;
  if (dtype == FLAREPP_BF16) {
    pl.tc = tc_plan(B, H, N, M, D, sms, g_forced_splits.load());
    pl.tiles = pl.tc.tiles;
    pl.splits = pl.tc.splits;
    pl.split_len = pl.tc.split_len;
    rows = (size_t)pl.BH * pl.tiles * pl.splits * pl.tc.streams * 128;
  } else {
    pl.tiles = (M + simt::kRows - 1) / simt::kRows;
    const int quantum = simt::kTile;
    const int max_splits = std::max(1, (N + quantum - 1) / quantum);
    int splits = g_forced_splits.load();
    if (splits <= 0) {
      const long long groups = (long long)pl.BH * pl.tiles;
      const long long want = std::max<long long>(1, (2LL * std::max(sms, 1) + groups - 1) / groups);
      splits = (int)std::min<long long>(want, 256);
    }
    splits = std::min(splits, max_splits);
    int split_len = (N + splits - 1) / splits;
    split_len = (split_len + quantum - 1) / quantum * quantum;
    pl.split_len = split_len;
    pl.splits = (N + split_len - 1) / split_len;
    rows = (size_t)pl.BH * pl.tiles * pl.splits * simt::kRows;
  }
  size_t off = 0;
  pl.off_pz = off; off = align_up(off + rows * D * sizeof(float), 256);
  pl.off_pl = off; off = align_up(off + rows * sizeof(float), 256);
  pl.off_cnt = off; off = align_up(off + 2 * (size_t)pl.BH * pl.tiles * sizeof(unsigned), 256);  // >= 2 BH qgroups
  const size_t lat = (size_t)pl.BH * M * D * elem_size(dtype);
  pl.off_q = off; off = align_up(off + lat, 256);
  pl.off_z = off; off = align_up(off + lat, 256);
  pl.total = off;
  return pl;
}

// bf16: the tensor-core kernels of tc.cu.
flarepp_status_t launch_tc(const Problem& p, const Plan& pl, char* ws, cudaStream_t stream) {
  unsigned* counters = reinterpret_cast<unsigned*>(ws + pl.off_cnt);
  if (!cuda_ok(cudaMemsetAsync(counters, 0, 2 * (size_t)pl.BH * pl.tiles * sizeof(unsigned), stream),
               "cudaMemsetAsync(counters)"))
    return FLAREPP_ERR_CUDA;
  DeviceProblem dp{};
  dp.variant = p.variant;
  dp.K = p.K; dp.V = p.V; dp.Ks = p.Ks; dp.Vs = p.Vs; dp.Qseed = p.Qseed; dp.Qf = p.Qf; dp.gate = p.gate;
  dp.Q = p.Q;
  dp.out = p.out;
  dp.B = p.B; dp.H = p.H; dp.N = p.N; dp.M = p.M; dp.D = p.D;
  dp.dbg_qd = p.dbg_qd; dp.dbg_q = p.dbg_q; dp.dbg_z = p.dbg_z; dp.dbg_l = p.dbg_l;
  dp.fail_wait = g_fail_wait.load();
  TcWorkspace w{};
  w.part_z = reinterpret_cast<float*>(ws + pl.off_pz);
  w.part_l = reinterpret_cast<float*>(ws + pl.off_pl);
  w.counters = counters;
  w.q = ws + pl.off_q;
  w.z = ws + pl.off_z;
  const char* failed = "";
  const cudaError_t e = tc_forward(dp, pl.tc, w, g_stage_events, stream, &failed);
  return cuda_ok(e, failed) ? FLAREPP_OK : FLAREPP_ERR_CUDA;
}

template <typename T, int D>
flarepp_status_t launch_typed(const Problem& p, const Plan& pl, char* ws, cudaStream_t stream) {
  Partials part;
  part.z = reinterpret_cast<float*>(ws + pl.off_pz);
  part.l = reinterpret_cast<float*>(ws + pl.off_pl);
  unsigned* counters = reinterpret_cast<unsigned*>(ws + pl.off_cnt);
  T* qbuf = reinterpret_cast<T*>(ws + pl.off_q);
  T* zbuf = reinterpret_cast<T*>(ws + pl.off_z);
  if (!cuda_ok(cudaMemsetAsync(counters, 0, 2 * (size_t)pl.BH * pl.tiles * sizeof(unsigned), stream),
               "cudaMemsetAsync(counters)"))
    return FLAREPP_ERR_CUDA;

  const dim3 grid(pl.splits, pl.tiles, pl.BH);
  const bool flare = p.variant == kVariantFlare;
  if (!stage_event(0, stream)) return FLAREPP_ERR_CUDA;
  simt::SplitArgs<T> sa{};
  sa.H = p.H; sa.N = p.N; sa.M = p.M;
  sa.tiles = pl.tiles; sa.splits = pl.splits; sa.split_len = pl.split_len;
  sa.part = part;
  if (!flare) {
    // synthesis: the variant's keys, values and queries (see launch.h)
    sa.keys = static_cast<const T*>(p.Ks);
    sa.values = static_cast<const T*>(p.variant == kVariantFlarePP ? p.Ks : p.Vs);
    sa.queries = static_cast<const T*>(p.Qseed);
    sa.q_by_head = 1;
    sa.part.counters = counters;
    sa.out = qbuf;
    if (p.variant == kVariantSimplified) {
      sa.dbg_a = p.dbg_q;  // Q = Qd, as rounded
      simt::split_kernel<T, D, kPassEncode><<<grid, simt::kRows, 0, stream>>>(sa);
    } else {
      sa.qf = static_cast<const T*>(p.Qf);
      sa.gate = p.gate;
      sa.dbg_a = p.dbg_qd;
      sa.dbg_b = p.dbg_q;
      if (p.variant == kVariantUnshared)
        simt::split_kernel<T, D, kPassSynthSeparate><<<grid, simt::kRows, 0, stream>>>(sa);
      else
        simt::split_kernel<T, D, kPassSynthShared><<<grid, simt::kRows, 0, stream>>>(sa);
    }
    if (!cuda_ok(cudaGetLastError(), "launch synthesis")) return FLAREPP_ERR_CUDA;
  }
  if (!stage_event(1, stream)) return FLAREPP_ERR_CUDA;

  // routing queries: FLARE's learned per-head set, or the synthesis output
  const T* qroute = flare ? static_cast<const T*>(p.Q) : qbuf;
  simt::SplitArgs<T> ea = sa;
  ea.keys = static_cast<const T*>(p.K);
  ea.values = static_cast<const T*>(p.V);
  ea.queries = qroute;
  ea.q_by_head = flare ? 1 : 0;
  ea.qf = nullptr;
  ea.gate = nullptr;
  ea.part.counters = counters + (size_t)pl.BH * pl.tiles;
  ea.out = zbuf;
  ea.dbg_a = p.dbg_z;
  ea.dbg_b = p.dbg_l;
  simt::split_kernel<T, D, kPassEncode><<<grid, simt::kRows, 0, stream>>>(ea);
  if (!cuda_ok(cudaGetLastError(), "launch encode")) return FLAREPP_ERR_CUDA;
  if (!stage_event(2, stream)) return FLAREPP_ERR_CUDA;

  simt::DecodeArgs<T> da;
  da.keys = static_cast<const T*>(p.K);
  da.q = qroute;
  da.z = zbuf;
  da.out = static_cast<T*>(p.out);
  da.N = p.N;
  da.M = p.M;
  da.H = p.H;
  da.q_by_head = flare ? 1 : 0;
  const size_t smem = 2 * (size_t)p.M * D * sizeof(float);
  if (!cuda_ok(cudaFuncSetAttribute(simt::decode_kernel<T, D>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
               "cudaFuncSetAttribute(decode)"))
    return FLAREPP_ERR_CUDA;
  const dim3 dgrid((p.N + simt::kDecodeTokens - 1) / simt::kDecodeTokens, pl.BH);
  simt::decode_kernel<T, D><<<dgrid, simt::kDecodeTokens, smem, stream>>>(da);
  if (!cuda_ok(cudaGetLastError(), "launch decode")) return FLAREPP_ERR_CUDA;
  if (!stage_event(3, stream)) return FLAREPP_ERR_CUDA;
  return FLAREPP_OK;
}

flarepp_status_t launch(const Problem& p, const Plan& pl, char* ws, cudaStream_t stream) {
  if (p.dtype == FLAREPP_FP32) {
    return p.D == 16 ? launch_typed<float, 16>(p, pl, ws, stream)
                     : launch_typed<float, 32>(p, pl, ws, stream);
  }
  return launch_tc(p, pl, ws, stream);
}

// Per-(device, stream) workspace cache, stream-ordered allocation. A caller
// holds g_cache_mu from the lookup until its kernels are enqueued: a thread
// that grows the buffer enqueues cudaFreeAsync of the old one on the stream,
// and a launch enqueued after that free must not use the old pointer.
struct CachedBuf {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::mutex g_cache_mu;
std::map<std::pair<int, cudaStream_t>, CachedBuf> g_cache;

// Caller holds g_cache_mu.
flarepp_status_t cached_workspace(size_t bytes, cudaStream_t stream, void** out) {
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev), "cudaGetDevice")) return FLAREPP_ERR_CUDA;
  CachedBuf& buf = g_cache[{dev, stream}];
  if (buf.bytes >= bytes) {
    *out = buf.ptr;
    return FLAREPP_OK;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (!cuda_ok(cudaStreamIsCapturing(stream, &cap), "cudaStreamIsCapturing")) return FLAREPP_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return FLAREPP_ERR_NO_MEMORY;  // grow outside capture
  if (buf.ptr != nullptr) {
    if (!cuda_ok(cudaFreeAsync(buf.ptr, stream), "cudaFreeAsync")) return FLAREPP_ERR_CUDA;
    buf.ptr = nullptr;
    buf.bytes = 0;
  }
  void* p = nullptr;
  const size_t want = align_up(bytes, 1 << 20);
  if (!cuda_ok(cudaMallocAsync(&p, want, stream), "cudaMallocAsync(workspace)")) {
    cudaGetLastError();
    return FLAREPP_ERR_NO_MEMORY;
  }
  buf.ptr = p;
  buf.bytes = want;
  *out = p;
  return FLAREPP_OK;
}

flarepp_status_t run(const Problem& p, void* workspace, size_t ws_bytes, bool use_cache,
                     cudaStream_t stream) {
  flarepp_status_t st = validate(p);
  if (st != FLAREPP_OK) return st;
  const int sms = device_sm_count();
  if (sms <= 0) {
    snprintf(g_last_error, sizeof(g_last_error), "no CUDA device (cudaGetDevice or attribute query failed)");
    return FLAREPP_ERR_CUDA;
  }
  const Plan pl = make_plan(p.B, p.H, p.N, p.M, p.D, p.dtype, sms);
  if (use_cache) {
    std::lock_guard<std::mutex> lock(g_cache_mu);  // until the kernels are enqueued
    st = cached_workspace(pl.total, stream, &workspace);
    if (st != FLAREPP_OK) return st;
    return launch(p, pl, static_cast<char*>(workspace), stream);
  }
  if (workspace == nullptr || ws_bytes < pl.total) return FLAREPP_ERR_NO_MEMORY;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FLAREPP_ERR_ALIGNMENT;
  return launch(p, pl, static_cast<char*>(workspace), stream);
}

Problem make_problem(const void* K, const void* V, const void* Ks, const void* Qseed, const void* Qf,
                     const float* gate, int B, int H, int N, int M, int D, flarepp_dtype_t dtype,
                     void* out) {
  Problem p{};
  p.K = K; p.V = V; p.Ks = Ks; p.Qseed = Qseed; p.Qf = Qf; p.gate = gate;
  p.B = B; p.H = H; p.N = N; p.M = M; p.D = D; p.dtype = dtype; p.out = out;
  return p;
}

}  // namespace
}  // namespace flarepp

using flarepp::Problem;

extern "C" {

flarepp_status_t flarepp_forward(const void* K, const void* V, const void* Ks_raw, const void* Qseed,
                                 const void* Qf, const float* gate, int B, int H, int N, int M, int D,
                                 flarepp_dtype_t dtype, void* out, cudaStream_t stream) {
  const Problem p = flarepp::make_problem(K, V, Ks_raw, Qseed, Qf, gate, B, H, N, M, D, dtype, out);
  return flarepp::run(p, nullptr, 0, true, stream);
}

size_t flarepp_workspace_size(int B, int H, int N, int M, int D, flarepp_dtype_t dtype) {
  if (flarepp::check_sizes(B, H, N, M, D, dtype) != FLAREPP_OK) return 0;
  const int sms = flarepp::device_sm_count();
  if (sms <= 0) return 0;
  return flarepp::make_plan(B, H, N, M, D, dtype, sms).total;
}

flarepp_status_t flarepp_plan_info(int B, int H, int N, int M, int D, flarepp_dtype_t dtype, int sms,
                                   int* fields, int n) {
  if (fields == nullptr || n < 1 || sms < 1) return FLAREPP_ERR_INVALID_ARG;
  const flarepp_status_t st = flarepp::check_sizes(B, H, N, M, D, dtype);
  if (st != FLAREPP_OK) return st;
  const flarepp::Plan pl = flarepp::make_plan(B, H, N, M, D, dtype, sms);
  const bool tc = dtype == FLAREPP_BF16;
  const long long v[8] = {pl.splits,
                          pl.split_len,
                          tc ? pl.tc.qgroups : 0,
                          tc ? pl.tc.decode_tiles_per_cta : 0,
                          tc ? pl.tc.decode_ctas_per_head : 0,
                          tc ? pl.tc.decode_heads : 0,
                          tc ? pl.tc.decode_ctas : 0,
                          (long long)std::min<size_t>(pl.total, (size_t)INT_MAX)};
  for (int i = 0; i < n && i < 8; ++i) fields[i] = (int)v[i];
  return FLAREPP_OK;
}

flarepp_status_t flarepp_forward_ws(const void* K, const void* V, const void* Ks_raw,
                                    const void* Qseed, const void* Qf, const float* gate, int B,
                                    int H, int N, int M, int D, flarepp_dtype_t dtype, void* out,
                                    void* workspace, size_t ws_bytes, cudaStream_t stream) {
  const Problem p = flarepp::make_problem(K, V, Ks_raw, Qseed, Qf, gate, B, H, N, M, D, dtype, out);
  return flarepp::run(p, workspace, ws_bytes, false, stream);
}

flarepp_status_t flarepp_forward_debug(const void* K, const void* V, const void* Ks_raw,
                                       const void* Qseed, const void* Qf, const float* gate, int B,
                                       int H, int N, int M, int D, flarepp_dtype_t dtype, void* out,
                                       float* Qd_out, float* Q_out, float* Z_out, float* L_out,
                                       cudaStream_t stream) {
  Problem p = flarepp::make_problem(K, V, Ks_raw, Qseed, Qf, gate, B, H, N, M, D, dtype, out);
  p.dbg_qd = Qd_out;
  p.dbg_q = Q_out;
  p.dbg_z = Z_out;
  p.dbg_l = L_out;
  return flarepp::run(p, nullptr, 0, true, stream);
}

flarepp_status_t flarepp_forward_variant(flarepp_variant_t variant, const void* K, const void* V,
                                         const void* Ks, const void* Vs, const void* Qseed,
                                         const void* Qf, const float* gate, int B, int H, int N,
                                         int M, int D, flarepp_dtype_t dtype, void* out,
                                         float* Qd_out, float* Q_out, float* Z_out, float* L_out,
                                         cudaStream_t stream) {
  if (variant != FLAREPP_VARIANT_SHARED && variant != FLAREPP_VARIANT_UNSHARED &&
      variant != FLAREPP_VARIANT_SIMPLIFIED)
    return FLAREPP_ERR_INVALID_ARG;
  Problem p = flarepp::make_problem(K, V, Ks, Qseed, Qf, gate, B, H, N, M, D, dtype, out);
  p.variant = variant == FLAREPP_VARIANT_SHARED     ? flarepp::kVariantFlarePP
              : variant == FLAREPP_VARIANT_UNSHARED ? flarepp::kVariantUnshared
                                                    : flarepp::kVariantSimplified;
  p.Vs = Vs;
  p.dbg_qd = variant == FLAREPP_VARIANT_SIMPLIFIED ? nullptr : Qd_out;
  p.dbg_q = Q_out;
  p.dbg_z = Z_out;
  p.dbg_l = L_out;
  return flarepp::run(p, nullptr, 0, true, stream);
}

flarepp_status_t flare_forward(const void* Q, const void* K, const void* V, int B, int H, int N, int M,
                               int D, flarepp_dtype_t dtype, void* out, float* Z_out, float* L_out,
                               cudaStream_t stream) {
  Problem p = flarepp::make_problem(K, V, nullptr, nullptr, nullptr, nullptr, B, H, N, M, D, dtype, out);
  p.variant = flarepp::kVariantFlare;
  p.Q = Q;
  p.dbg_z = Z_out;
  p.dbg_l = L_out;
  return flarepp::run(p, nullptr, 0, true, stream);
}

flarepp_status_t flarepp_project(const void* X, const void* W, const float* bias, int P,
                                 const flarepp_norm_t* norms, const float* scales, void* const* outs,
                                 int B, int H, int N, int D, flarepp_dtype_t dtype,
                                 cudaStream_t stream) {
  using flarepp::overlaps;
  if (B <= 0 || H <= 0 || N <= 0 || D <= 0 || P < 1 || P > flarepp::kMaxProjParts)
    return FLAREPP_ERR_INVALID_ARG;
  if (X == nullptr || W == nullptr || norms == nullptr || outs == nullptr) return FLAREPP_ERR_INVALID_ARG;
  if (dtype != FLAREPP_BF16 && dtype != FLAREPP_FP32) return FLAREPP_ERR_UNSUPPORTED;
  const bool bf16 = dtype == FLAREPP_BF16;
  if (!flarepp::proj_supported(H, D, bf16)) return FLAREPP_ERR_UNSUPPORTED;
  if ((long long)B * H * N * D >= (1LL << 31) || B > 65535) return FLAREPP_ERR_UNSUPPORTED;
  flarepp::ProjProblem pp{};
  bool any_na = false;
  for (int i = 0; i < P; ++i) {
    if (norms[i] != FLAREPP_NORM_NONE && norms[i] != FLAREPP_NORM_N0 && norms[i] != FLAREPP_NORM_NA)
      return FLAREPP_ERR_INVALID_ARG;
    if (outs[i] == nullptr) return FLAREPP_ERR_INVALID_ARG;
    any_na = any_na || norms[i] == FLAREPP_NORM_NA;
    pp.norms[i] = static_cast<int>(norms[i]);
    pp.outs[i] = outs[i];
  }
  if (any_na != (scales != nullptr)) return FLAREPP_ERR_INVALID_ARG;
  const void* ptrs[] = {X, W, bias, scales};
  for (const void* q : ptrs)
    if (q != nullptr && (reinterpret_cast<uintptr_t>(q) & 15u) != 0) return FLAREPP_ERR_ALIGNMENT;
  for (int i = 0; i < P; ++i)
    if ((reinterpret_cast<uintptr_t>(outs[i]) & 15u) != 0) return FLAREPP_ERR_ALIGNMENT;
  const size_t es = bf16 ? 2 : 4;
  const size_t C = (size_t)H * D;
  const size_t out_bytes = (size_t)B * N * C * es;
  const std::pair<const void*, size_t> ins[] = {{X, out_bytes},
                                                {W, (size_t)P * C * C * es},
                                                {bias, (size_t)P * C * 4},
                                                {scales, (size_t)P * D * 4}};
  for (int i = 0; i < P; ++i) {
    for (const auto& in : ins)
      if (in.first != nullptr && overlaps(outs[i], out_bytes, in.first, in.second)) return FLAREPP_ERR_INVALID_ARG;
    for (int k = 0; k < i; ++k)
      if (overlaps(outs[i], out_bytes, outs[k], out_bytes)) return FLAREPP_ERR_INVALID_ARG;
  }
  const int sms = flarepp::device_sm_count();
  if (sms <= 0) {
    snprintf(flarepp::g_last_error, sizeof(flarepp::g_last_error), "no CUDA device");
    return FLAREPP_ERR_CUDA;
  }
  pp.X = X;
  pp.W = W;
  pp.bias = bias;
  pp.scales = scales;
  pp.P = P;
  pp.B = B;
  pp.H = H;
  pp.N = N;
  pp.D = D;
  const char* failed = "";
  const cudaError_t e = flarepp::proj_forward(pp, sms, bf16, stream, &failed);
  return flarepp::cuda_ok(e, failed) ? FLAREPP_OK : FLAREPP_ERR_CUDA;
}

flarepp_status_t flarepp_backward(const void* K, const void* V, const void* Ks_raw, const void* Qseed,
                                  const void* Qf, const float* gate, const void* dY, int B, int H, int N,
                                  int M, int D, flarepp_dtype_t dtype, float* dK, float* dV, float* dKs_raw,
                                  float* dQseed, float* dQf, float* dgate, cudaStream_t stream) {
  using flarepp::overlaps;
  flarepp_status_t st = flarepp::check_sizes(B, H, N, M, D, dtype);
  if (st != FLAREPP_OK) return st;
  const void* req[] = {K, V, Ks_raw, Qseed, Qf, gate, dY, dK, dV, dKs_raw, dQseed, dQf, dgate};
  for (const void* q : req) {
    if (q == nullptr) return FLAREPP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0) return FLAREPP_ERR_ALIGNMENT;
  }
  const size_t es = dtype == FLAREPP_BF16 ? 2 : 4;
  const size_t tok = (size_t)B * H * N * D, lat = (size_t)H * M * D;
  const std::pair<const void*, size_t> ins[] = {{K, tok * es},     {V, tok * es},   {Ks_raw, tok * es},
                                                {Qseed, lat * es}, {Qf, lat * es},  {gate, (size_t)H * 4},
                                                {dY, tok * es}};
  const std::pair<const void*, size_t> outs[] = {{dK, tok * 4},     {dV, tok * 4},  {dKs_raw, tok * 4},
                                                 {dQseed, lat * 4}, {dQf, lat * 4}, {dgate, (size_t)H * 4}};
  for (size_t i = 0; i < 6; ++i) {
    for (const auto& in : ins)
      if (overlaps(outs[i].first, outs[i].second, in.first, in.second)) return FLAREPP_ERR_INVALID_ARG;
    for (size_t k = 0; k < i; ++k)
      if (overlaps(outs[i].first, outs[i].second, outs[k].first, outs[k].second)) return FLAREPP_ERR_INVALID_ARG;
  }
  const int sms = flarepp::device_sm_count();
  if (sms <= 0) {
    snprintf(flarepp::g_last_error, sizeof(flarepp::g_last_error), "no CUDA device");
    return FLAREPP_ERR_CUDA;
  }
  const bool bf16 = dtype == FLAREPP_BF16;
  void* ws = nullptr;
  std::lock_guard<std::mutex> lock(flarepp::g_cache_mu);  // until the kernels are enqueued
  st = flarepp::cached_workspace(flarepp::backward_workspace_bytes(B, H, N, M, D, bf16, sms), stream, &ws);
  if (st != FLAREPP_OK) return st;
  flarepp::BwdProblem p{};
  p.K = K; p.V = V; p.Ks = Ks_raw; p.Qseed = Qseed; p.Qf = Qf; p.gate = gate; p.dY = dY;
  p.B = B; p.H = H; p.N = N; p.M = M; p.D = D; p.bf16 = bf16;
  p.dK = dK; p.dV = dV; p.dKs = dKs_raw; p.dQseed = dQseed; p.dQf = dQf; p.dgate = dgate;
  const char* failed = "";
  const cudaError_t e = flarepp::backward_run(p, ws, flarepp::backward_workspace_bytes(B, H, N, M, D, bf16, sms),
                                              sms, stream, &failed);
  return flarepp::cuda_ok(e, failed) ? FLAREPP_OK : FLAREPP_ERR_CUDA;
}

flarepp_status_t flarepp_sync_status(cudaStream_t stream) {
  using flarepp::cuda_ok;
  if (!cuda_ok(cudaStreamSynchronize(stream), "cudaStreamSynchronize")) return FLAREPP_ERR_CUDA;
  unsigned word = 0;
  if (!cuda_ok(cudaMemcpyFromSymbol(&word, flarepp::g_error_word, sizeof(word)), "read error word"))
    return FLAREPP_ERR_CUDA;
  if (word != 0) {
    const unsigned zero = 0;
    if (!cuda_ok(cudaMemcpyToSymbol(flarepp::g_error_word, &zero, sizeof(zero)), "clear error word"))
      return FLAREPP_ERR_CUDA;
  }
  unsigned tc_word = 0, proj_word = 0;
  if (!cuda_ok(flarepp::tc_take_error_word(&tc_word), "read tensor-core error word")) return FLAREPP_ERR_CUDA;
  if (!cuda_ok(flarepp::proj_take_error_word(&proj_word), "read projection error word")) return FLAREPP_ERR_CUDA;
  word |= tc_word | proj_word;
  if (word != 0) {
    snprintf(flarepp::g_last_error, sizeof(flarepp::g_last_error), "device error word 0x%x", word);
    return (word & flarepp::kErrTimeout) ? FLAREPP_ERR_TIMEOUT : FLAREPP_ERR_CUDA;
  }
  return FLAREPP_OK;
}

const char* flarepp_status_string(flarepp_status_t status) {
  switch (status) {
    case FLAREPP_OK: return "ok";
    case FLAREPP_ERR_INVALID_ARG: return "invalid argument";
    case FLAREPP_ERR_UNSUPPORTED: return "unsupported size or dtype";
    case FLAREPP_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case FLAREPP_ERR_NO_MEMORY: return "workspace unavailable or too small";
    case FLAREPP_ERR_CUDA: return "CUDA error";
    case FLAREPP_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* flarepp_last_error(void) { return flarepp::g_last_error; }

void flarepp_set_splits(int splits) { flarepp::g_forced_splits.store(splits < 0 ? 0 : splits); }

void flarepp_test_fail_wait(int pass) { flarepp::g_fail_wait.store(pass >= 1 && pass <= 3 ? pass : 0); }

flarepp_status_t flarepp_debug_trace(int pass, unsigned long long* host, int n) {
  const cudaError_t e = flarepp::tc_trace(pass, host, n);
  if (e == cudaErrorNotSupported) return FLAREPP_ERR_UNSUPPORTED;
  return flarepp::cuda_ok(e, "pipeline trace") ? FLAREPP_OK : FLAREPP_ERR_CUDA;
}

void flarepp_set_stage_events(cudaEvent_t* events, int count) {
  flarepp::g_stage_events = (events != nullptr && count >= 4) ? events : nullptr;
}

}  // extern "C"
