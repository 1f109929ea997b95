// Tensor-core (tcgen05 + TMEM + TMA) kernels of the FLARE++ mixer forward,
// bf16 inputs, fp32 softmax and accumulation.
//
// Two kernels carry the three attention calls of the mixer (FLARE++ paper,
// Section 3.2 eq. 6 and eq. 8):
//
//  * split_kernel — a 128-row block of latent queries attends over one token
//    range (split) of a head: scores S = Qtile * Ktile^T land in TMEM, one
//    thread per latent row runs an online softmax over the tokens, P goes back
//    to TMEM in bf16 and the tensor core accumulates O += P * Vtile in TMEM.
//    The split's (Z_s, L_s) go to global memory and the last CTA of the head to
//    arrive merges all splits with the stable log-sum-exp schedule of
//    Appendix B.3 (eq. 29-33). The synthesis instance normalises each staged
//    Ks_raw tile in place (N0, eq. 5), uses it as both keys and values
//    (eq. 19) and ends with the gate (eq. 7): Q = N0(Qf) + g * Qd in fp32, cast
//    to bf16. The encode instance ends with Z (bf16) and L.
//  * decode_kernel — 128 tokens per tile attend over the M routes: Q and Z of
//    the head stay in shared memory for all of the CTA's tiles, scores
//    S = Ktile * Q^T are computed 128 routes at a time, softmax over M per
//    token (one thread per token), Y += P * Z in TMEM, then Y / l to bf16.
//
// Warp roles (256 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs (one thread), warps 2-3 normalise synthesis tiles, warps
// 4-7 run the softmax and the epilogues; warp 4+i reads TMEM lanes 32i..32i+31.
//
// Every wait on an mbarrier is bounded: after about a second without progress
// the thread records kErrTimeout in the device error word, raises the CTA's
// abort flag and leaves its loop, so a broken invariant ends the kernel
// instead of hanging the GPU.
#include <cuda.h>
#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"

namespace flarepp {
namespace tc {

using namespace sm100;

__device__ unsigned g_tc_error = 0u;

constexpr int kThreads = 256;
constexpr int kTile = 128;      // tokens per staged tile; latents per row block
constexpr int kStages = 4;      // token-tile ring depth
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;    // fp32 scores, 128 columns
constexpr uint32_t kColP = 128;  // bf16 probabilities, 64 columns (128 packed pairs)
constexpr uint32_t kColO = 192;  // fp32 output accumulator, D columns
constexpr long long kWaitLimit = 2000000000LL;  // clock cycles (~1 s)
constexpr size_t kMinSmem = 80 * 1024;          // keeps residency at <= 2 CTAs per SM

struct Shared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t norm[kStages];
  uint64_t q_full;
  uint64_t s_full;
  uint64_t p_full;
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int last;
};

__device__ __forceinline__ bool wait_or_abort(Shared& sh, uint64_t* bar, uint32_t parity) {
  if (*(volatile int*)&sh.abort) return false;
  if (mbar_wait(bar, parity, kWaitLimit)) return true;
  atomicOr(&g_tc_error, kErrTimeout);
  *(volatile int*)&sh.abort = 1;
  return false;
}

__device__ __forceinline__ void named_sync_softmax() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

template <int D>
struct Layout {
  static constexpr uint32_t kRowBytes = D * 2;
  static constexpr uint32_t kAtom = 8 * kRowBytes;          // one swizzle repeat (8 rows)
  static constexpr uint32_t kTileBytes = kTile * kRowBytes;  // 128 rows
  static constexpr uint32_t kSwz = D == 32 ? kSwizzle64 : kSwizzle32;
  // K-major operand (rows x D), k-th 16-element slice
  static __device__ __forceinline__ uint64_t kmajor(uint32_t base, int k) {
    return sdesc(base + k * 32, 16, kAtom, kSwz);
  }
  // MN-major operand: rows are the K dimension, D columns the N dimension;
  // slice kk covers rows 16kk .. 16kk+15
  static __device__ __forceinline__ uint64_t mnmajor(uint32_t base, int kk) {
    return sdesc(base + kk * 2 * kAtom, 16, kAtom, kSwz);
  }
};

// exp2 of x <= 0 (or slightly above after a lazy max): MUFU ex2.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Scales the D accumulator columns of this thread's TMEM lane by `alpha`.
template <int D>
__device__ __forceinline__ void rescale_acc(uint32_t taddr, float alpha) {
  uint32_t r[16];
#pragma unroll
  for (int c = 0; c < D; c += 16) {
    tmem_ld16(taddr + c, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
    tmem_st16(taddr + c, r);
  }
  tmem_wait_st();
}

template <int D>
__device__ __forceinline__ void load_acc(uint32_t taddr, float (&o)[D]) {
  uint32_t r[16];
#pragma unroll
  for (int c = 0; c < D; c += 16) {
    tmem_ld16(taddr + c, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) o[c + i] = __uint_as_float(r[i]);
  }
}

// One softmax step over `width` (multiple of 16, <= 128) score columns of this
// thread's TMEM lane, columns >= `valid` masked out. Keeps the running max
// `m` (raw score units) and sum `l`; rescales the accumulator lazily, only
// when the max grows by more than 2^8 in exp2 units, so p <= 256 always.
// Writes P (bf16 pairs) to the P columns. `has_acc`: the accumulator holds
// earlier steps' products.
template <int D>
__device__ __forceinline__ void softmax_step(uint32_t tS, uint32_t tP, uint32_t tO, int width, int valid,
                                             float c, float& m, float& l, bool has_acc) {
  constexpr float kLazy = 8.0f;
  float tmax = -INFINITY;
  for (int base = 0; base < width; base += 32) {
    uint32_t r[32];
    if (width - base >= 32) {
      tmem_ld32(tS + base, r);
    } else {
      uint32_t h[16];
      tmem_ld16(tS + base, h);
#pragma unroll
      for (int i = 0; i < 16; ++i) { r[i] = h[i]; r[16 + i] = __float_as_uint(-INFINITY); }
    }
    tmem_wait_ld();
    if (valid - base >= 32) {
#pragma unroll
      for (int i = 0; i < 32; i += 2)
        tmax = fmaxf(tmax, fmaxf(__uint_as_float(r[i]), __uint_as_float(r[i + 1])));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (base + i < valid) tmax = fmaxf(tmax, __uint_as_float(r[i]));
    }
  }
  // the max moves only when it grows by more than 2^8 (in exp2 units); TMEM
  // access is warp-collective, so the warp rescales together (alpha = 1 for
  // lanes whose max stays)
  const bool grow = tmax > m && (m == -INFINITY || (tmax - m) * c > kLazy);
  float alpha = 1.f;
  if (grow) {
    alpha = m == -INFINITY ? 0.f : ex2((m - tmax) * c);
    l *= alpha;
    m = tmax;
  }
  if (has_acc && __any_sync(0xFFFFFFFFu, grow)) rescale_acc<D>(tO, alpha);
  const float mc = m * c;
  for (int base = 0; base < width; base += 32) {
    uint32_t r[32];
    const bool full = width - base >= 32;
    if (full) {
      tmem_ld32(tS + base, r);
    } else {
      uint32_t h[16];
      tmem_ld16(tS + base, h);
#pragma unroll
      for (int i = 0; i < 16; ++i) { r[i] = h[i]; r[16 + i] = 0u; }
    }
    tmem_wait_ld();
    uint32_t pk[16];
    if (valid - base >= 32) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = ex2(fmaf(__uint_as_float(r[2 * i]), c, -mc));
        const float p1 = ex2(fmaf(__uint_as_float(r[2 * i + 1]), c, -mc));
        l += p0 + p1;
        pk[i] = pack_bf16(p0, p1);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = base + 2 * i < valid ? ex2(fmaf(__uint_as_float(r[2 * i]), c, -mc)) : 0.f;
        const float p1 = base + 2 * i + 1 < valid ? ex2(fmaf(__uint_as_float(r[2 * i + 1]), c, -mc)) : 0.f;
        l += p0 + p1;
        pk[i] = pack_bf16(p0, p1);
      }
    }
    if (full) {
      tmem_st16(tP + base / 2, pk);
    } else {
      // 16 score columns -> 8 packed columns
      uint32_t a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = pk[i];
      tmem_st8(tP + base / 2, a);
    }
  }
  tmem_wait_st();
}

// ------------------------------------------------------------ split kernel
struct SplitParams {
  int N, M, H, tiles, splits, split_len, streams;
  float* part_z;
  float* part_l;
  unsigned* counters;
  const __nv_bfloat16* qf;  // synthesis: [H][M][D]
  const float* gate;        // synthesis: [H]
  __nv_bfloat16* out;       // synthesis: Q; encode: Z ([BH][M][D])
  float* dbg_a;             // synthesis: Qd; encode: Z (as rounded)
  float* dbg_b;             // synthesis: Q (as rounded); encode: L
};

template <int D, bool kSynth>
__global__ void __launch_bounds__(kThreads, 2)
    split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const SplitParams p) {
  using L = Layout<D>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ Shared sh;
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  constexpr uint32_t kStageBytes = kSynth ? L::kTileBytes : 2 * L::kTileBytes;
  unsigned char* sQ = smem;
  unsigned char* sStage = smem + 8192;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x, tile = blockIdx.y, bh = blockIdx.z;
  const int h = bh % p.H;
  const bool two = p.streams == 2;
  const int n_begin = split * p.split_len;
  const int n_end = min(p.N, n_begin + p.split_len);
  const int T = n_begin < n_end ? (n_end - n_begin + kTile - 1) / kTile : 0;  // token tiles
  const int steps = two ? (T + 1) / 2 : T;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
      mbar_init(&sh.norm[s], 64);
    }
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.p_full, 128);
    mbar_init(&sh.o_full, 1);
    mbar_init(&sh.drain, 1);
    sh.abort = 0;
    sh.last = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      if (!kSynth) prefetch_tmap(&tm_v);
      const int qz = kSynth ? h : bh;
      if (two) {
        mbar_arrive_expect_tx(&sh.q_full, L::kTileBytes);
        tma_load_3d(sQ, &tm_q, &sh.q_full, 0, 0, qz);
        tma_load_3d(sQ + L::kTileBytes / 2, &tm_q, &sh.q_full, 0, 0, qz);
      } else {
        mbar_arrive_expect_tx(&sh.q_full, L::kTileBytes);
        tma_load_3d(sQ, &tm_q, &sh.q_full, 0, tile * kTile, qz);
      }
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % kStages;
        if (t >= kStages && !wait_or_abort(sh, &sh.empty[s], ((t / kStages) - 1) & 1)) break;
        unsigned char* dst = sStage + s * kStageBytes;
        mbar_arrive_expect_tx(&sh.full[s], kStageBytes);
        tma_load_3d(dst, &tm_k, &sh.full[s], 0, n_begin + t * kTile, bh);
        if (!kSynth) tma_load_3d(dst + L::kTileBytes, &tm_v, &sh.full[s], 0, n_begin + t * kTile, bh);
        issued = t + 1;
      }
      if (*(volatile int*)&sh.abort) {
        // let the copies still in flight land before the CTA leaves
        for (int t = max(0, issued - kStages); t < issued; ++t)
          mbar_wait(&sh.full[t % kStages], (t / kStages) & 1, kWaitLimit);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t aQ = smem_u32(sQ);
      const uint32_t idS = idesc_bf16(128, kTile, false, false);
      const uint32_t idO = idesc_bf16(128, D, false, true);
      bool ok = wait_or_abort(sh, &sh.q_full, 0);
      for (int j = 0; ok && j < steps; ++j) {
        const int ta = two ? 2 * j : j;
        const bool has_b = two && (2 * j + 1 < T);
        const int sa = ta % kStages, sb = (ta + 1) % kStages;
        uint64_t* ready_a = kSynth ? &sh.norm[sa] : &sh.full[sa];
        uint64_t* ready_b = kSynth ? &sh.norm[sb] : &sh.full[sb];
        if (!wait_or_abort(sh, ready_a, (ta / kStages) & 1)) break;
        if (has_b && !wait_or_abort(sh, ready_b, ((ta + 1) / kStages) & 1)) break;
        tc_fence_after();
        const uint32_t kA = smem_u32(sStage + sa * kStageBytes);
        const uint32_t kB = smem_u32(sStage + sb * kStageBytes);
        if (!two) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss(tmem + kColS, L::kmajor(aQ, k), L::kmajor(kA, k), idS, k > 0);
        } else {
          // rows 0-63 score the even tile, rows 64-127 (same latents) the odd one
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss_masked(tmem + kColS, L::kmajor(aQ, k), L::kmajor(kA, k), idS, k > 0, 0u, 0u,
                          0xFFFFFFFFu, 0xFFFFFFFFu);
          if (has_b) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_ss_masked(tmem + kColS, L::kmajor(aQ, k), L::kmajor(kB, k), idS, k > 0, 0xFFFFFFFFu,
                            0xFFFFFFFFu, 0u, 0u);
          }
        }
        mma_commit(&sh.s_full);
        if (!wait_or_abort(sh, &sh.p_full, j & 1)) break;
        tc_fence_after();
        const uint32_t vA = kSynth ? kA : kA + L::kTileBytes;
        const uint32_t vB = kSynth ? kB : kB + L::kTileBytes;
        if (!two) {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts(tmem + kColO, tmem + kColP + kk * 8, L::mnmajor(vA, kk), idO, (j > 0 || kk > 0));
        } else {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts_masked(tmem + kColO, tmem + kColP + kk * 8, L::mnmajor(vA, kk), idO, (j > 0 || kk > 0),
                          0u, 0u, 0xFFFFFFFFu, 0xFFFFFFFFu);
          if (has_b) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ts_masked(tmem + kColO, tmem + kColP + kk * 8, L::mnmajor(vB, kk), idO,
                            (j > 0 || kk > 0), 0xFFFFFFFFu, 0xFFFFFFFFu, 0u, 0u);
          }
        }
        mma_commit(&sh.empty[sa]);
        if (has_b) mma_commit(&sh.empty[sb]);
      }
      mma_commit(&sh.o_full);
      // all MMAs of this CTA complete before TMEM is released
      mma_commit(&sh.drain);
      mbar_wait(&sh.drain, 0, kWaitLimit);
    }
  } else if (warp < 4) {
    // ------------------------------------------- N0 of the synthesis tiles
    if (kSynth) {
      const int nt = threadIdx.x - 64;  // 0..63, rows nt and nt + 64
      for (int t = 0; t < T; ++t) {
        const int s = t % kStages;
        if (!wait_or_abort(sh, &sh.full[s], (t / kStages) & 1)) break;
        unsigned char* tileb = sStage + s * kStageBytes;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint4* row = reinterpret_cast<uint4*>(tileb + (nt + 64 * half) * L::kRowBytes);
          uint4 v[D / 8];
          float ss = 0.f;
#pragma unroll
          for (int i = 0; i < D / 8; ++i) {
            v[i] = row[i];
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float a = __uint_as_float(w[j] << 16), b = __uint_as_float(w[j] & 0xFFFF0000u);
              ss = fmaf(a, a, fmaf(b, b, ss));
            }
          }
          const float r = rsqrtf(ss / (float)D + kEps);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) {
            uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
              w[j] = pack_bf16(__uint_as_float(w[j] << 16) * r, __uint_as_float(w[j] & 0xFFFF0000u) * r);
            row[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&sh.norm[s]);
      }
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int row = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + kColS;
    const uint32_t tP = tmem + lane_base + kColP;
    const uint32_t tO = tmem + lane_base + kColO;
    const int stream = two ? (row >> 6) : 0;
    const int r_in = two ? (row & 63) : row;
    const int latent = tile * kTile + r_in;
    const bool valid = latent < p.M;
    const float c = rsqrtf((float)D) * kLog2e;
    float m = -INFINITY, l = 0.f;
    bool has_acc = false;
    bool ok = true;
    for (int j = 0; j < steps; ++j) {
      if (!wait_or_abort(sh, &sh.s_full, j & 1)) { ok = false; break; }
      tc_fence_after();
      const int t = two ? 2 * j + stream : j;
      if (t < T) {
        const int n0 = n_begin + t * kTile;
        softmax_step<D>(tS, tP, tO, kTile, min(kTile, n_end - n0), c, m, l, has_acc);
        has_acc = true;
      }
      // (a stream with no tile in the last step skips it: its lanes of the
      // two masked products are neither computed into S nor accumulated)
      tc_fence_before();
      mbar_arrive(&sh.p_full);
    }
    if (ok) ok = wait_or_abort(sh, &sh.o_full, 0);
    tc_fence_after();
    float o[D];
    load_acc<D>(tO, o);
    const int streams_total = p.splits * p.streams;
    const size_t grp = (size_t)bh * p.tiles + tile;
    if (valid) {
      const size_t prow = (grp * streams_total + (size_t)split * p.streams + stream) * kTile + r_in;
      float z[D];
      const bool any = ok && l > 0.f;  // a stream with no token never wrote its accumulator
      const float inv = any ? 1.f / l : 0.f;
#pragma unroll
      for (int d = 0; d < D; ++d) z[d] = any ? o[d] * inv : 0.f;
      store_row<D>(p.part_z + prow * D, z);
      p.part_l[prow] = any ? (m * c + __log2f(l)) * kLn2 : -INFINITY;
    }
    __threadfence();
    named_sync_softmax();
    if (row == 0) {
      const unsigned prev = atomicAdd(p.counters + grp, 1u);
      sh.last = prev == (unsigned)(p.splits - 1);
    }
    named_sync_softmax();
    if (sh.last) {
      __threadfence();
      if (row == 0) p.counters[grp] = 0u;  // ready for the next call
      const bool merges = valid && (!two || row < 64);
      if (merges) {
        // Appendix B.3: L_max, d_s = exp(L_s - L_max), U = sum d_s Z_s, Z = U / d
        const size_t p0 = grp * streams_total * kTile + r_in;
        float lmax = -INFINITY;
        for (int s = 0; s < streams_total; ++s) lmax = fmaxf(lmax, __ldcg(p.part_l + p0 + (size_t)s * kTile));
        float u[D], dsum = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) u[d] = 0.f;
        for (int s = 0; s < streams_total; ++s) {
          const size_t r = p0 + (size_t)s * kTile;
          const float ls = __ldcg(p.part_l + r);
          if (ls == -INFINITY) continue;
          const float w = __expf(ls - lmax);
          dsum += w;
          const float4* zr = reinterpret_cast<const float4*>(p.part_z + r * D);
#pragma unroll
          for (int d = 0; d < D; d += 4) {
            const float4 zz = __ldcg(zr + d / 4);
            u[d] = fmaf(w, zz.x, u[d]);
            u[d + 1] = fmaf(w, zz.y, u[d + 1]);
            u[d + 2] = fmaf(w, zz.z, u[d + 2]);
            u[d + 3] = fmaf(w, zz.w, u[d + 3]);
          }
        }
        const float invd = 1.f / dsum;
#pragma unroll
        for (int d = 0; d < D; ++d) u[d] *= invd;
        const size_t orow = (size_t)bh * p.M + latent;
        if (kSynth) {
          // gate (eq. 7): Q = N0(Qf) + g * Qd in fp32, cast to bf16
          float f[D];
          load_row<D>(p.qf + ((size_t)h * p.M + latent) * D, f);
          float ss = 0.f;
#pragma unroll
          for (int d = 0; d < D; ++d) ss = fmaf(f[d], f[d], ss);
          const float rr = rsqrtf(ss / (float)D + kEps);
          const float g = p.gate[h];
          float q[D];
#pragma unroll
          for (int d = 0; d < D; ++d) q[d] = fmaf(g, u[d], f[d] * rr);
          store_row<D>(p.out + orow * D, q);
          if (p.dbg_a) store_row<D>(p.dbg_a + orow * D, u);
          if (p.dbg_b) {
#pragma unroll
            for (int d = 0; d < D; ++d) q[d] = round_as<__nv_bfloat16>(q[d]);
            store_row<D>(p.dbg_b + orow * D, q);
          }
        } else {
          store_row<D>(p.out + orow * D, u);
          if (p.dbg_a) {
#pragma unroll
            for (int d = 0; d < D; ++d) u[d] = round_as<__nv_bfloat16>(u[d]);
            store_row<D>(p.dbg_a + orow * D, u);
          }
          if (p.dbg_b) p.dbg_b[orow] = lmax + __logf(dsum);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ----------------------------------------------------------- decode kernel
struct DecodeParams {
  int N, M, tiles_per_cta;
  __nv_bfloat16* out;  // [BH][N][D]
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_z, const DecodeParams p) {
  using L = Layout<D>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ Shared sh;
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  const int chunks = (p.M + kTile - 1) / kTile;
  unsigned char* sQ = smem;                                // [chunks][128][D]
  unsigned char* sZ = smem + chunks * L::kTileBytes;       // [chunks][128][D]
  unsigned char* sK = smem + 2 * chunks * L::kTileBytes;   // [kStages][128][D]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int n_tiles = (p.N + kTile - 1) / kTile;
  const int t_begin = blockIdx.x * p.tiles_per_cta;
  const int T = max(0, min(n_tiles, t_begin + p.tiles_per_cta) - t_begin);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.p_full, 128);
    mbar_init(&sh.o_full, 1);
    mbar_init(&sh.drain, 1);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_z);
      mbar_arrive_expect_tx(&sh.q_full, 2 * chunks * L::kTileBytes);
      for (int ch = 0; ch < chunks; ++ch) {
        tma_load_3d(sQ + ch * L::kTileBytes, &tm_q, &sh.q_full, 0, ch * kTile, bh);
        tma_load_3d(sZ + ch * L::kTileBytes, &tm_z, &sh.q_full, 0, ch * kTile, bh);
      }
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % kStages;
        if (t >= kStages && !wait_or_abort(sh, &sh.empty[s], ((t / kStages) - 1) & 1)) break;
        mbar_arrive_expect_tx(&sh.full[s], L::kTileBytes);
        tma_load_3d(sK + s * L::kTileBytes, &tm_k, &sh.full[s], 0, (t_begin + t) * kTile, bh);
        issued = t + 1;
      }
      if (*(volatile int*)&sh.abort) {
        for (int t = max(0, issued - kStages); t < issued; ++t)
          mbar_wait(&sh.full[t % kStages], (t / kStages) & 1, kWaitLimit);
        mbar_wait(&sh.q_full, 0, kWaitLimit);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t aQ = smem_u32(sQ), aZ = smem_u32(sZ);
      const uint32_t idO = idesc_bf16(128, D, false, true);
      bool ok = wait_or_abort(sh, &sh.q_full, 0);
      int step = 0;
      for (int t = 0; ok && t < T; ++t) {
        const int s = t % kStages;
        if (!wait_or_abort(sh, &sh.full[s], (t / kStages) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t aK = smem_u32(sK + s * L::kTileBytes);
        for (int ch = 0; ch < chunks; ++ch, ++step) {
          const int width = min(kTile, p.M - ch * kTile);
          const uint32_t idS = idesc_bf16(128, width, false, false);
          const uint32_t qc = aQ + ch * L::kTileBytes;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) mma_ss(tmem + kColS, L::kmajor(aK, k), L::kmajor(qc, k), idS, k > 0);
          if (ch == chunks - 1) mma_commit(&sh.empty[s]);
          mma_commit(&sh.s_full);
          if (!wait_or_abort(sh, &sh.p_full, step & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t zc = aZ + ch * L::kTileBytes;
          for (int kk = 0; kk < width / 16; ++kk)
            mma_ts(tmem + kColO, tmem + kColP + kk * 8, L::mnmajor(zc, kk), idO, (ch > 0 || kk > 0));
          if (ch == chunks - 1) mma_commit(&sh.o_full);
        }
      }
      mma_commit(&sh.drain);
      mbar_wait(&sh.drain, 0, kWaitLimit);
    }
  } else if (warp >= 4) {
    const int row = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + kColS;
    const uint32_t tP = tmem + lane_base + kColP;
    const uint32_t tO = tmem + lane_base + kColO;
    const float c = rsqrtf((float)D) * kLog2e;
    int step = 0;
    for (int t = 0; t < T; ++t) {
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int ch = 0; ch < chunks; ++ch, ++step) {
        if (!wait_or_abort(sh, &sh.s_full, step & 1)) { ok = false; break; }
        tc_fence_after();
        const int width = min(kTile, p.M - ch * kTile);
        softmax_step<D>(tS, tP, tO, width, width, c, m, l, ch > 0);
        tc_fence_before();
        mbar_arrive(&sh.p_full);
      }
      if (!ok) break;
      if (!wait_or_abort(sh, &sh.o_full, t & 1)) break;
      tc_fence_after();
      float y[D];
      load_acc<D>(tO, y);
      const int n = (t_begin + t) * kTile + row;
      if (n < p.N) {
        const float inv = 1.f / l;
#pragma unroll
        for (int d = 0; d < D; ++d) y[d] *= inv;
        store_row<D>(p.out + ((size_t)bh * p.N + n) * D, y);
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 3-D map over a [planes][rows][D] bf16 tensor, box {D, box_rows, 1}, swizzled
// to the row width (64 B for D = 32, 32 B for D = 16). Rows past `rows` of a
// plane read as zero.
bool make_map(CUtensorMap* map, const void* base, int D, int rows, int planes, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * rows};
  const cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz = D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
size_t split_smem(bool synth) {
  const size_t stage = synth ? Layout<D>::kTileBytes : 2 * Layout<D>::kTileBytes;
  const size_t need = 1024 + 8192 + kStages * stage;
  return need < kMinSmem ? kMinSmem : need;
}

template <int D>
size_t decode_smem(int M) {
  const int chunks = (M + kTile - 1) / kTile;
  const size_t need = 1024 + (2 * chunks + kStages) * (size_t)Layout<D>::kTileBytes;
  return need < kMinSmem ? kMinSmem : need;
}

template <int D>
cudaError_t forward_d(const DeviceProblem& pr, const TcPlan& pl, const TcWorkspace& ws, cudaEvent_t* ev,
                      cudaStream_t stream, const char** failed) {
  const int BH = pr.B * pr.H;
  cudaError_t e;
  CUtensorMap m_seed, m_ks, m_qbuf, m_k, m_v, m_qdec, m_zdec;
  const int qbox = pl.streams == 2 ? 64 : kTile;
  *failed = "cuTensorMapEncodeTiled";
  if (!make_map(&m_seed, pr.Qseed, D, pr.M, pr.H, qbox) || !make_map(&m_ks, pr.Ks, D, pr.N, BH, kTile) ||
      !make_map(&m_qbuf, ws.q, D, pr.M, BH, qbox) || !make_map(&m_k, pr.K, D, pr.N, BH, kTile) ||
      !make_map(&m_v, pr.V, D, pr.N, BH, kTile) || !make_map(&m_qdec, ws.q, D, pr.M, BH, kTile) ||
      !make_map(&m_zdec, ws.z, D, pr.M, BH, kTile))
    return cudaErrorInvalidValue;

  const dim3 grid(pl.splits, pl.tiles, BH);
  SplitParams sp{};
  sp.N = pr.N; sp.M = pr.M; sp.H = pr.H;
  sp.tiles = pl.tiles; sp.splits = pl.splits; sp.split_len = pl.split_len; sp.streams = pl.streams;
  sp.part_z = ws.part_z; sp.part_l = ws.part_l;

  if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) { *failed = "cudaEventRecord"; return e; }
  // synthesis (a1-a3)
  {
    SplitParams a = sp;
    a.counters = ws.counters;
    a.qf = static_cast<const __nv_bfloat16*>(pr.Qf);
    a.gate = pr.gate;
    a.out = static_cast<__nv_bfloat16*>(ws.q);
    a.dbg_a = pr.dbg_qd;
    a.dbg_b = pr.dbg_q;
    const size_t smem = split_smem<D>(true);
    *failed = "cudaFuncSetAttribute(synthesis)";
    if ((e = cudaFuncSetAttribute(split_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    split_kernel<D, true><<<grid, kThreads, smem, stream>>>(m_seed, m_ks, m_ks, a);
    *failed = "launch synthesis";
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) { *failed = "cudaEventRecord"; return e; }
  // encode (a4-a5)
  {
    SplitParams a = sp;
    a.counters = ws.counters + (size_t)BH * pl.tiles;
    a.out = static_cast<__nv_bfloat16*>(ws.z);
    a.dbg_a = pr.dbg_z;
    a.dbg_b = pr.dbg_l;
    const size_t smem = split_smem<D>(false);
    *failed = "cudaFuncSetAttribute(encode)";
    if ((e = cudaFuncSetAttribute(split_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    split_kernel<D, false><<<grid, kThreads, smem, stream>>>(m_qbuf, m_k, m_v, a);
    *failed = "launch encode";
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (ev && (e = cudaEventRecord(ev[2], stream)) != cudaSuccess) { *failed = "cudaEventRecord"; return e; }
  // decode (a6)
  {
    DecodeParams d{};
    d.N = pr.N; d.M = pr.M; d.tiles_per_cta = pl.decode_tiles_per_cta;
    d.out = static_cast<__nv_bfloat16*>(pr.out);
    const size_t smem = decode_smem<D>(pr.M);
    *failed = "cudaFuncSetAttribute(decode)";
    if ((e = cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    decode_kernel<D><<<dim3(pl.decode_ctas_per_head, BH), kThreads, smem, stream>>>(m_k, m_qdec, m_zdec, d);
    *failed = "launch decode";
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (ev && (e = cudaEventRecord(ev[3], stream)) != cudaSuccess) { *failed = "cudaEventRecord"; return e; }
  *failed = "";
  return cudaSuccess;
}

}  // namespace tc

TcPlan tc_plan(int B, int H, int N, int M, int D, int sms, int forced_splits) {
  (void)D;
  TcPlan pl{};
  const long long BH = (long long)B * H;
  pl.streams = M <= 64 ? 2 : 1;
  pl.tiles = pl.streams == 2 ? 1 : (M + tc::kTile - 1) / tc::kTile;
  const int n_tiles = (N + tc::kTile - 1) / tc::kTile;
  // about two CTAs per SM for each split-N pass, each split a whole number of
  // token tiles (an even number in the two-stream mode)
  const int quantum = pl.streams;  // tiles per split step
  int splits = forced_splits;
  if (splits <= 0) {
    const long long groups = BH * pl.tiles;
    splits = (int)std::min<long long>(256, std::max<long long>(1, (2LL * sms + groups - 1) / groups));
  }
  const int max_splits = std::max(1, (n_tiles + quantum - 1) / quantum);
  splits = std::min(splits, max_splits);
  int tiles_per_split = (n_tiles + splits - 1) / splits;
  tiles_per_split = (tiles_per_split + quantum - 1) / quantum * quantum;
  pl.split_len = tiles_per_split * tc::kTile;
  pl.splits = (N + pl.split_len - 1) / pl.split_len;
  // decode: enough CTAs for two per SM, each reusing the head's Q and Z over
  // consecutive token tiles
  const long long want = std::max<long long>(1, (2LL * sms + BH - 1) / BH);
  const int per = (int)std::max<long long>(1, (n_tiles + want - 1) / want);
  pl.decode_tiles_per_cta = per;
  pl.decode_ctas_per_head = (n_tiles + per - 1) / per;
  return pl;
}

cudaError_t tc_forward(const DeviceProblem& p, const TcPlan& pl, const TcWorkspace& ws, cudaEvent_t* events,
                       cudaStream_t stream, const char** failed_call) {
  return p.D == 16 ? tc::forward_d<16>(p, pl, ws, events, stream, failed_call)
                   : tc::forward_d<32>(p, pl, ws, events, stream, failed_call);
}

cudaError_t tc_take_error_word(unsigned* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, tc::g_tc_error, sizeof(unsigned));
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(tc::g_tc_error, &zero, sizeof(unsigned));
}

}  // namespace flarepp
