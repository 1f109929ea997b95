// Fused token projections that produce the FLARE++ mixer's inputs (FLARE++
// paper, Section 3.2 and Appendix A.7 Table 2): for P stacked projections
//
//   out_p[b, h, n, :] = norm_p( X[b, n, :] W_p^T + bias_p )[h*D : h*D + D]
//
// with norm_p one of: none, N0 (RMSNorm over D without scale) or N_a (RMSNorm
// over D with a learned scale of D values shared by the heads). For the
// default mixer: K = N_a(X W_K), V = X W_V and the raw synthesis keys X W~_K.
//
// At the widths of the paper's models (C = H D <= 256) a projection moves
// 2C bytes in and 2C bytes out per token for 2C^2 flops, about C/2 flops per
// byte, so it is bound by HBM, not by the tensor core. The kernel is therefore
// built to read X once and write each output once, at full bandwidth:
//
//  * persistent CTAs (one per SM) walk 128-token tiles of one batch entry;
//    each tile of X ([128, C] bf16) is loaded by TMA into one of two buffers,
//    a whole tile ahead of its use;
//  * the weights stream through a ring of [128 output channels, 64 inputs]
//    stages (they stay in L2; every tile reads them again from there);
//  * one thread issues the tcgen05 MMAs (M = 128 tokens, N = 128 channels,
//    K = 16) into four 128-column TMEM accumulators, so the tensor core fills
//    the next chunks while the epilogue drains one;
//  * epilogue warps in groups of four (one per TMEM lane quarter), each group
//    taking 32 or 64 channels of every chunk, add the bias, normalise each head's D values, round to bf16, write the
//    head tiles [128 tokens, D] into shared memory in the swizzled layout of
//    the mixer's token tiles, and TMA-store them straight into [B, H, N, D];
//    rows past N are clipped by the store.
//
// The fp32 verification build has a plain CUDA-core kernel (one thread per
// token and head).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"
#include "tmap.h"

namespace flarepp {
namespace proj {

using namespace sm100;

__device__ unsigned g_proj_error = 0u;

constexpr int kTok = 128;        // tokens per tile (MMA M, TMEM lanes)
constexpr int kWarpX = 0;        // lane 0: TMA loads of X tiles
constexpr int kWarpMma = 1;      // lane 0: MMA issue; the warp owns TMEM
constexpr int kWarpW = 2;        // lane 0: TMA loads of weight stages
constexpr int kWarpEpi = 4;      // epilogue warps 4-11
constexpr int kAccBufs = 4;      // TMEM accumulators
constexpr long long kWaitLimit = 2000000000LL;  // clock cycles (~1 s)

template <int D, int C>
struct Cfg {
  static constexpr int kKc = C / 64;                    // 64-element input chunks (128-byte rows)
  static constexpr int kChunk = C >= 128 ? 128 : 64;    // output channels per accumulator
  // channels per epilogue group (4 warps): at C = 256 two groups of 64, so
  // that fewer epilogue warps compete for issue slots with the MMA thread,
  // whose issue rate bounds that width; otherwise groups of 32
  static constexpr int kGroupCh = C == 256 ? 64 : 32;
  static constexpr int kGroups = kChunk / kGroupCh;     // epilogue groups (4 warps each)
  static constexpr int kHeadsGroup = kGroupCh / D;      // whole heads per group
  static constexpr int kThreads = 32 * kWarpEpi + 128 * kGroups;
  static constexpr uint32_t kXChunkBytes = kTok * 128;  // [128 tokens, 64 inputs]
  static constexpr uint32_t kXBytes = kKc * kXChunkBytes;
  static constexpr uint32_t kWStageBytes = kChunk * 128;
  static constexpr int kWStages = C == 256 ? 3 : 7;  // as deep as shared memory allows
  static constexpr uint32_t kHeadTileBytes = kTok * D * 2;
  static constexpr uint32_t kStageOutBytes = kHeadsGroup * kHeadTileBytes;
  static constexpr uint32_t kParamFloats = kMaxProjParts * (C + D);  // bias and N_a scales
  static constexpr uint32_t kTmemCols = kAccBufs * kChunk;
  static constexpr size_t kSmem = 1024 + 2 * (size_t)kXBytes + kWStages * (size_t)kWStageBytes +
                                  kGroups * (size_t)kStageOutBytes + kParamFloats * 4;
  static_assert(C % 64 == 0 && C <= 256, "C = H D must be 64, 128 or 256");
  static_assert(kGroupCh % D == 0, "an epilogue group holds whole heads");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct Bars {
  uint64_t x_full[2], x_empty[2];
  uint64_t w_full[8], w_empty[8];
  uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool wait_or_abort(Bars& sh, uint64_t* bar, uint32_t parity) {
  if (*(volatile int*)&sh.abort) return false;
  if (mbar_wait(bar, parity, kWaitLimit)) return true;
  atomicOr(&g_proj_error, kErrTimeout);
  *(volatile int*)&sh.abort = 1;
  return false;
}

// One arrival per warp once the warp's TMEM loads are complete.
__device__ __forceinline__ void warp_arrive_acc(uint64_t* bar) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Byte offset of 16-byte chunk `c` of row `r` in a [128, D] head tile, in the
// layout the TMA maps of the token tensors use (32-byte swizzle at D = 16,
// 64-byte at D = 32).
template <int D>
__device__ __forceinline__ uint32_t head_chunk_offset(int r, int c) {
  const int x = D == 32 ? ((r >> 1) & 3) : ((r >> 2) & 1);
  return r * (D * 2) + ((c ^ x) << 4);
}

struct OutMaps {
  CUtensorMap m[kMaxProjParts];
};

template <int D, int C>
__global__ void __launch_bounds__(Cfg<D, C>::kThreads, 1)
    proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ OutMaps tm_out, const ProjParams p) {
  using G = Cfg<D, C>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ Bars sh;
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  unsigned char* sX = smem;                                    // [2][kKc][128 x 128 B]
  unsigned char* sW = sX + 2 * G::kXBytes;                     // [kWStages][kChunk x 128 B]
  unsigned char* sOut = sW + G::kWStages * G::kWStageBytes;    // [groups][heads][128 x D]
  float* sBias = reinterpret_cast<float*>(sOut + G::kGroups * G::kStageOutBytes);  // [P*C]
  float* sScale = sBias + kMaxProjParts * C;                                       // [P][D]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles =
      p.tiles > (int)blockIdx.x ? (p.tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int n_chunks = p.P * C / G::kChunk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.x_full[i], 1);
      mbar_init(&sh.x_empty[i], 1);
    }
    for (int i = 0; i < G::kWStages; ++i) {
      mbar_init(&sh.w_full[i], 1);
      mbar_init(&sh.w_empty[i], 1);
    }
    for (int i = 0; i < kAccBufs; ++i) {
      mbar_init(&sh.acc_full[i], 1);
      mbar_init(&sh.acc_empty[i], 4 * G::kGroups);  // one arrival per epilogue warp
    }
    mbar_init(&sh.drain, 1);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sh.tmem_base, G::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == kWarpX) {
    // ----------------------------------------------------------- X tiles
    if (lane == 0) {
      prefetch_tmap(&tm_x);
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int buf = i & 1;
        if (i >= 2 && !wait_or_abort(sh, &sh.x_empty[buf], ((i >> 1) - 1) & 1)) break;
        const int t = blockIdx.x + i * gridDim.x;
        const int b = t / p.tiles_per_b, j = t % p.tiles_per_b;
        mbar_arrive_expect_tx(&sh.x_full[buf], G::kXBytes);
        for (int kc = 0; kc < G::kKc; ++kc)
          tma_load_3d(sX + buf * G::kXBytes + kc * G::kXChunkBytes, &tm_x, &sh.x_full[buf], 64 * kc, j * kTok, b);
        issued = i + 1;
      }
      if (*(volatile int*)&sh.abort) {
        // let the copies still in flight land before the CTA leaves
        for (int i = std::max(0, issued - 2); i < issued; ++i) mbar_wait(&sh.x_full[i & 1], (i >> 1) & 1, kWaitLimit);
      }
    }
  } else if (warp == kWarpW) {
    // ----------------------------------------------------- weight stages
    if (lane == 0) {
      prefetch_tmap(&tm_w);
      int it = 0;
      bool ok = true;
      for (int i = 0; ok && i < n_tiles; ++i)
        for (int c = 0; ok && c < n_chunks; ++c)
          for (int kc = 0; ok && kc < G::kKc; ++kc) {
            const int s = it % G::kWStages;
            if (it >= G::kWStages && !wait_or_abort(sh, &sh.w_empty[s], ((it / G::kWStages) - 1) & 1)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sh.w_full[s], G::kWStageBytes);
            tma_load_2d(sW + s * G::kWStageBytes, &tm_w, &sh.w_full[s], 64 * kc, c * G::kChunk);
            ++it;
          }
      if (*(volatile int*)&sh.abort) {
        for (int k = std::max(0, it - G::kWStages); k < it; ++k)
          mbar_wait(&sh.w_full[k % G::kWStages], (k / G::kWStages) & 1, kWaitLimit);
      }
    }
  } else if (warp == kWarpMma) {
    // -------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kTok, G::kChunk, false, false);
      // K-major operands, 128-byte rows in 128-byte swizzle: 8-row groups
      // 1024 bytes apart; a 16-element step along K is 32 bytes (2 units)
      const uint64_t dX0 = sdesc(smem_u32(sX), 16, 1024, kSwizzle128);
      const uint64_t dW0 = sdesc(smem_u32(sW), 16, 1024, kSwizzle128);
      int it = 0, cit = 0;
      bool ok = true;
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int buf = i & 1;
        if (!wait_or_abort(sh, &sh.x_full[buf], (i >> 1) & 1)) break;
        tc_fence_after();
        for (int c = 0; ok && c < n_chunks; ++c, ++cit) {
          const int a = cit % kAccBufs;
          if (cit >= kAccBufs && !wait_or_abort(sh, &sh.acc_empty[a], ((cit / kAccBufs) - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dAcc = tmem + a * G::kChunk;
          for (int kc = 0; kc < G::kKc; ++kc, ++it) {
            const int s = it % G::kWStages;
            if (!wait_or_abort(sh, &sh.w_full[s], (it / G::kWStages) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ax = dX0 + ((buf * G::kXBytes + kc * G::kXChunkBytes) >> 4);
            const uint64_t bw = dW0 + ((s * G::kWStageBytes) >> 4);
#pragma unroll
            for (int q = 0; q < 4; ++q) mma_ss(dAcc, ax + 2 * q, bw + 2 * q, idesc, (kc | q) ? 1u : 0u);
            mma_commit(&sh.w_empty[s]);
          }
          if (ok) mma_commit(&sh.acc_full[a]);
        }
        mma_commit(&sh.x_empty[buf]);
      }
      // every MMA of this CTA completes before TMEM is released
      mma_commit(&sh.drain);
      mbar_wait(&sh.drain, 0, kWaitLimit);
    }
  } else if (warp >= kWarpEpi) {
    // --------------------------------------------------------- epilogue
    const int g = (warp - kWarpEpi) >> 2;  // 32-channel group of every chunk
    const int qd = warp & 3;               // TMEM lane quarter
    const int row = 32 * qd + lane;        // token within the tile
    const bool leader = warp == kWarpEpi + 4 * g && lane == 0;  // issues the group's stores
    unsigned char* stage = sOut + g * G::kStageOutBytes;
    const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
    // the bias and the N_a scales, once per CTA (0 and 1 where absent)
    const int etid = threadIdx.x - 32 * kWarpEpi;
    for (int e = etid; e < p.P * C; e += 128 * G::kGroups) sBias[e] = p.bias != nullptr ? p.bias[e] : 0.f;
    for (int e = etid; e < p.P * D; e += 128 * G::kGroups) sScale[e] = p.scales != nullptr ? p.scales[e] : 1.f;
    named_bar_sync(15, 128 * G::kGroups);
    int cit = 0;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int t = blockIdx.x + i * gridDim.x;
      const int b = t / p.tiles_per_b, j = t % p.tiles_per_b;
      for (int c = 0; c < n_chunks; ++c, ++cit) {
        const int a = cit % kAccBufs;
        ok = ok && wait_or_abort(sh, &sh.acc_full[a], (cit / kAccBufs) & 1);
        tc_fence_after();
        uint32_t v[G::kGroupCh];
        if (ok) {
          const uint32_t src = tmem + lane_base + a * G::kChunk + g * G::kGroupCh;
          if constexpr (G::kGroupCh == 64) {
            tmem_ld64(src, v);
          } else {
            tmem_ld32(src, v);
          }
          tmem_wait_ld_regs(v);
        }
        warp_arrive_acc(&sh.acc_empty[a]);
        // the group's staging buffer is free once its previous stores have read it
        if (leader) bulk_wait_group_read<0>();
        named_bar_sync(1 + g, 128);
        const int o0 = c * G::kChunk + g * G::kGroupCh;  // first output channel of the group
        const int part = o0 / C;
        const int h0 = (o0 % C) / D;
        if (ok) {
          // select by comparison: a dynamic index into the parameter array
          // would copy it to local memory
          int norm = p.norms[0];
#pragma unroll
          for (int q = 1; q < kMaxProjParts; ++q)
            if (part == q) norm = p.norms[q];
#pragma unroll
          for (int hh = 0; hh < G::kHeadsGroup; ++hh) {
            float x[D];
            const float4* bq = reinterpret_cast<const float4*>(sBias + o0 + hh * D);
#pragma unroll
            for (int d = 0; d < D; d += 4) {
              const float4 bb = bq[d / 4];
              x[d] = __uint_as_float(v[hh * D + d]) + bb.x;
              x[d + 1] = __uint_as_float(v[hh * D + d + 1]) + bb.y;
              x[d + 2] = __uint_as_float(v[hh * D + d + 2]) + bb.z;
              x[d + 3] = __uint_as_float(v[hh * D + d + 3]) + bb.w;
            }
            if (norm != kNormNone) {
              float ss = 0.f;
#pragma unroll
              for (int d = 0; d < D; ++d) ss = fmaf(x[d], x[d], ss);
              const float r = rsqrtf(ss / (float)D + kEps);
              if (norm == kNormNa) {
                const float4* sq = reinterpret_cast<const float4*>(sScale + part * D);
#pragma unroll
                for (int d = 0; d < D; d += 4) {
                  const float4 a4 = sq[d / 4];
                  x[d] *= r * a4.x;
                  x[d + 1] *= r * a4.y;
                  x[d + 2] *= r * a4.z;
                  x[d + 3] *= r * a4.w;
                }
              } else {
#pragma unroll
                for (int d = 0; d < D; ++d) x[d] *= r;
              }
            }
            unsigned char* tile = stage + hh * G::kHeadTileBytes;
#pragma unroll
            for (int cc = 0; cc < D / 8; ++cc) {
              const uint4 w = make_uint4(pack_bf16x2(x[8 * cc], x[8 * cc + 1]), pack_bf16x2(x[8 * cc + 2], x[8 * cc + 3]),
                                         pack_bf16x2(x[8 * cc + 4], x[8 * cc + 5]),
                                         pack_bf16x2(x[8 * cc + 6], x[8 * cc + 7]));
              *reinterpret_cast<uint4*>(tile + head_chunk_offset<D>(row, cc)) = w;
            }
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1 + g, 128);
        if (leader && ok) {
          const CUtensorMap* m = &tm_out.m[part];
#pragma unroll
          for (int hh = 0; hh < G::kHeadsGroup; ++hh)
            tma_store_3d(m, stage + hh * G::kHeadTileBytes, 0, j * kTok, b * p.H + h0 + hh);
          bulk_commit_group();
        }
      }
    }
    if (leader) bulk_wait_group<0>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, G::kTmemCols);
}

// ------------------------------------------------------------ fp32 build
// One thread per (token, head, projection): D dot products of length C over
// the token's row of X (staged in shared memory for 32 tokens), then the bias
// and the head's norm.
constexpr int kSimtTokens = 32;
constexpr int kSimtThreads = 256;

template <int D>
__global__ void __launch_bounds__(kSimtThreads)
    proj_simt_kernel(const float* __restrict__ X, const float* __restrict__ W, ProjParams p, int C,
                     float* o0, float* o1, float* o2, float* o3) {
  extern __shared__ float xs[];  // [kSimtTokens][C]
  const int b = blockIdx.y;
  const int n0 = blockIdx.x * kSimtTokens;
  const int cnt = min(kSimtTokens, p.N - n0);
  for (int e = threadIdx.x; e < cnt * C; e += blockDim.x) xs[e] = X[((size_t)b * p.N + n0) * C + e];
  __syncthreads();
  float* outs[kMaxProjParts] = {o0, o1, o2, o3};
  const int units = cnt * p.H * p.P;
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    const int tok = u % cnt;
    const int h = (u / cnt) % p.H;
    const int part = u / (cnt * p.H);
    float y[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int o = part * C + h * D + d;
      const float* w = W + (size_t)o * C;
      const float* x = xs + tok * C;
      float acc = 0.f;
      for (int k = 0; k < C; ++k) acc = fmaf(x[k], __ldg(w + k), acc);
      y[d] = acc + (p.bias != nullptr ? p.bias[o] : 0.f);
    }
    const int norm = p.norms[part];
    if (norm != kNormNone) {
      float ss = 0.f;
#pragma unroll
      for (int d = 0; d < D; ++d) ss = fmaf(y[d], y[d], ss);
      const float r = rsqrtf(ss / (float)D + kEps);
#pragma unroll
      for (int d = 0; d < D; ++d) y[d] *= norm == kNormNa ? r * p.scales[part * D + d] : r;
    }
    store_row<D>(outs[part] + (((size_t)b * p.H + h) * p.N + n0 + tok) * D, y);
  }
}

// ------------------------------------------------------------------ host
template <int D, int C>
cudaError_t launch_tc(const ProjProblem& pp, const ProjParams& prm, int sms, cudaStream_t stream,
                      const char** failed) {
  using G = Cfg<D, C>;
  CUtensorMap mx, mw;
  OutMaps mo;
  *failed = "cuTensorMapEncodeTiled";
  {
    const cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)pp.N, (cuuint64_t)pp.B};
    const cuuint64_t strides[2] = {(cuuint64_t)C * 2, (cuuint64_t)C * 2 * pp.N};
    const cuuint32_t box[3] = {64, (cuuint32_t)kTok, 1};
    if (!make_map_bf16(&mx, pp.X, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)pp.P * C};
    const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)G::kChunk};
    if (!make_map_bf16(&mw, pp.W, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }
  for (int i = 0; i < kMaxProjParts; ++i) {
    const void* base = pp.outs[i < pp.P ? i : 0];
    if (!make_map(&mo.m[i], base, D, pp.N, pp.B * pp.H, kTok)) return cudaErrorInvalidValue;
  }
  *failed = "cudaFuncSetAttribute(proj_kernel)";
  cudaError_t e = cudaFuncSetAttribute(proj_kernel<D, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)G::kSmem);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(prm.tiles, sms));
  proj_kernel<D, C><<<grid, G::kThreads, G::kSmem, stream>>>(mx, mw, mo, prm);
  *failed = "launch proj_kernel";
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_tc_d(const ProjProblem& pp, const ProjParams& prm, int sms, cudaStream_t stream,
                        const char** failed) {
  const int C = pp.H * D;
  if (C == 64) return launch_tc<D, 64>(pp, prm, sms, stream, failed);
  if (C == 128) return launch_tc<D, 128>(pp, prm, sms, stream, failed);
  return launch_tc<D, 256>(pp, prm, sms, stream, failed);
}

template <int D>
cudaError_t launch_simt(const ProjProblem& pp, const ProjParams& prm, cudaStream_t stream, const char** failed) {
  const int C = pp.H * D;
  float* o[kMaxProjParts];
  for (int i = 0; i < kMaxProjParts; ++i) o[i] = static_cast<float*>(pp.outs[i < pp.P ? i : 0]);
  const size_t smem = (size_t)kSimtTokens * C * sizeof(float);
  *failed = "cudaFuncSetAttribute(proj_simt_kernel)";
  cudaError_t e = cudaFuncSetAttribute(proj_simt_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((pp.N + kSimtTokens - 1) / kSimtTokens, pp.B);
  proj_simt_kernel<D><<<grid, kSimtThreads, smem, stream>>>(static_cast<const float*>(pp.X),
                                                           static_cast<const float*>(pp.W), prm, C, o[0],
                                                           o[1], o[2], o[3]);
  *failed = "launch proj_simt_kernel";
  return cudaGetLastError();
}

}  // namespace proj

bool proj_supported(int H, int D, bool bf16) {
  if (D != 16 && D != 32) return false;
  const int C = H * D;
  return bf16 ? (C == 64 || C == 128 || C == 256) : C <= 256;
}

cudaError_t proj_forward(const ProjProblem& pp, int sms, bool bf16, cudaStream_t stream, const char** failed) {
  ProjParams prm{};
  prm.N = pp.N;
  prm.H = pp.H;
  prm.P = pp.P;
  prm.tiles_per_b = (pp.N + proj::kTok - 1) / proj::kTok;
  prm.tiles = prm.tiles_per_b * pp.B;
  prm.bias = pp.bias;
  prm.scales = pp.scales;
  for (int i = 0; i < kMaxProjParts; ++i) prm.norms[i] = i < pp.P ? pp.norms[i] : kNormNone;
  if (bf16)
    return pp.D == 16 ? proj::launch_tc_d<16>(pp, prm, sms, stream, failed)
                      : proj::launch_tc_d<32>(pp, prm, sms, stream, failed);
  return pp.D == 16 ? proj::launch_simt<16>(pp, prm, stream, failed)
                    : proj::launch_simt<32>(pp, prm, stream, failed);
}

cudaError_t proj_take_error_word(unsigned* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, proj::g_proj_error, sizeof(unsigned));
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(proj::g_proj_error, &zero, sizeof(unsigned));
}

}  // namespace flarepp
