// Tensor-core (tcgen05 + TMEM + TMA) kernels of the FLARE++ mixer forward,
// bf16 inputs, fp32 softmax and accumulation.
//
// Two kernels carry the three attention calls of the mixer (FLARE++ paper,
// Section 3.2 eq. 6 and eq. 8):
//
//  * split_kernel — latent queries attend over one token range (split) of a
//    head. Scores S = Q K^T land in TMEM; one thread per latent row runs an
//    online softmax over the tokens; P goes back to TMEM in bf16 over the
//    scores and the tensor core accumulates O += P [V | 1] in TMEM, the
//    appended ones column giving the softmax row sum. Each split's (Z_s, L_s)
//    goes to global memory and the last CTA of a head to arrive merges all
//    splits with the stable log-sum-exp schedule of Appendix B.3 (eq. 29-33).
//    The synthesis instance normalises each staged Ks_raw tile in place (N0,
//    eq. 5), uses it as both keys and values (eq. 19) and ends with the gate
//    (eq. 7): Q = N0(Qf) + g * Qd in fp32, cast to bf16. The encode instance
//    ends with Z (bf16) and L.
//  * decode_kernel — tokens attend over the M routes: Q and Z of the head stay
//    in shared memory for all of the CTA's token tiles; S = K Q^T is computed
//    128 routes at a time with an online softmax over M per token, and
//    O += P [Z | 1]; out = O / rowsum in bf16.
//
// One CTA per SM, 384 threads: warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs (one thread), warps 2-3 normalise synthesis tiles, and two
// softmax warpgroups (warps 4-7 and 8-11) each own one of two TMEM slots, so
// one slot's softmax runs while the tensor core works on the other's products.
// Warp w reads TMEM lanes 32*(w%4) .. +31.
//
// Every wait on an mbarrier is bounded: after about a second without progress
// the thread records kErrTimeout in the device error word, raises the CTA's
// abort flag and leaves its loop, so a broken invariant ends the kernel
// instead of hanging the GPU.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"

namespace flarepp {
namespace tc {

using namespace sm100;

__device__ unsigned g_tc_error = 0u;

constexpr int kThreads = 384;
constexpr int kTile = 128;          // tokens per staged tile; latents per row block
constexpr int kStages = 6;          // token-tile ring depth
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSlotCols = 256;  // slot s: scores at s*256, accumulator at +128, probabilities at +176
constexpr uint32_t kColO = 128;
constexpr uint32_t kColP = 176;
constexpr long long kWaitLimit = 2000000000LL;  // clock cycles (~1 s)

// How the two TMEM slots of a split-kernel CTA divide the work:
//  kLanes   (M <= 64)  each slot holds the latents twice; lanes 0-63 and 64-127
//                      score different token tiles (4 token streams per CTA);
//  kStreams            one 128-row latent block, the slots take alternate tiles;
//  kPair               two 128-row latent blocks, both slots see every tile.
enum : int { kLanes = 0, kStreams = 1, kPair = 2 };

struct Shared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t norm[kStages];
  uint64_t q_full;
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
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

// Barrier over the two softmax warpgroups only (256 threads).
__device__ __forceinline__ void softmax_groups_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int D>
struct Layout {
  static constexpr uint32_t kRowBytes = D * 2;
  static constexpr uint32_t kAtom = 8 * kRowBytes;           // one swizzle repeat (8 rows)
  static constexpr uint32_t kTileBytes = kTile * kRowBytes;  // 128 rows
  static constexpr uint32_t kSwz = D == 32 ? kSwizzle64 : kSwizzle32;
  static constexpr int kNo = D + 16;  // accumulator columns: D values, the row sum, padding
  // K-major operand (rows x D), k-th 16-element slice
  static __device__ __forceinline__ uint64_t kmajor(uint32_t base, int k) {
    return sdesc(base + k * 32, 16, kAtom, kSwz);
  }
  // MN-major [values | ones] operand: rows are the K dimension; the D value
  // columns sit at `base`, the ones column block `ones - base` bytes further.
  // Slice kk covers rows 16kk .. 16kk+15.
  static __device__ __forceinline__ uint64_t values1(uint32_t base, uint32_t ones, int kk) {
    return sdesc(base + kk * 2 * kAtom, ones - base, kAtom, kSwz);
  }
  // Byte offset of logical 16-byte chunk `c` of row `r` in a swizzled tile.
  static __device__ __forceinline__ uint32_t chunk_offset(int r, int c) {
    const int x = D == 32 ? ((r >> 1) & 3) : ((r >> 2) & 1);
    return r * kRowBytes + ((c ^ x) << 4);
  }
};

// Fills a 128-row tile, in the swizzled layout of the value tiles, with rows
// [1, 0, ..., 0]: as the extra column block of an MN-major B operand it makes
// the MMA add the probabilities of each row into accumulator column D.
template <int D>
__device__ void fill_ones(unsigned char* tile, int tid, int nthreads) {
  using L = Layout<D>;
  for (int i = tid; i < kTile * (D / 8); i += nthreads) {
    const int r = i / (D / 8), c = i % (D / 8);
    const uint4 v = make_uint4(c == 0 ? 0x3F80u : 0u, 0u, 0u, 0u);  // bf16 1.0 in element 0
    *reinterpret_cast<uint4*>(tile + L::chunk_offset(r, c)) = v;
  }
}

// Scales the accumulator columns (values and row sum) of this lane by `alpha`.
template <int D>
__device__ __forceinline__ void rescale_acc(uint32_t taddr, float alpha) {
  uint32_t r[16];
#pragma unroll
  for (int c = 0; c < Layout<D>::kNo; c += 16) {
    tmem_ld16(taddr + c, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
    tmem_st16(taddr + c, r);
  }
  tmem_wait_st();
}

// Reads the D output values and the row sum of this lane's accumulator.
template <int D>
__device__ __forceinline__ float load_acc(uint32_t taddr, float (&o)[D]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  if (D == 32) {
    uint32_t s[16];
    tmem_ld16(taddr + 32, s);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < D; ++i) o[i] = __uint_as_float(r[i]);
    return __uint_as_float(s[0]);
  }
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < D; ++i) o[i] = __uint_as_float(r[i]);
  return __uint_as_float(r[D]);
}

// One softmax step over `kWidth` (32, 64 or 128) score columns of this lane,
// columns >= `valid` masked. `m` is the running max in raw score units; it
// moves only when the tile max exceeds it by more than 2^8 in exp2 units
// (then the accumulator, row sum included, is rescaled), so p <= 256. P is
// written in bf16 to the kWidth/2 probability columns at tP. The scores are
// read twice (max, then exponentials), 64 columns at a time, to keep the
// live registers low. Warp-uniform: every lane of a warp calls it with the
// same width and valid count.
template <int D, int kWidth>
__device__ __forceinline__ void softmax_step(uint32_t tS, uint32_t tP, uint32_t tO, int valid, float c,
                                             float& m, bool has_acc) {
  constexpr float kLazy = 8.0f;
  constexpr int kPart = kWidth < 64 ? kWidth : 64;
  float tmax = m;
#pragma unroll
  for (int base = 0; base < kWidth; base += kPart) {
    uint32_t r[kPart];
#pragma unroll
    for (int b = 0; b < kPart; b += 32) tmem_ld32(tS + base + b, *reinterpret_cast<uint32_t(*)[32]>(r + b));
    tmem_wait_ld();
    if (valid < base + kPart) {
#pragma unroll
      for (int i = 0; i < kPart; ++i)
        if (base + i >= valid) r[i] = __float_as_uint(-INFINITY);
    }
#pragma unroll
    for (int i = 0; i < kPart; i += 2) tmax = max3(tmax, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
  }
  const bool grow = tmax > m && (m == -INFINITY || (tmax - m) * c > kLazy);
  float alpha = 1.f;
  if (grow) {
    alpha = m == -INFINITY ? 0.f : ex2((m - tmax) * c);
    m = tmax;
  }
  if (has_acc && __any_sync(0xFFFFFFFFu, grow)) rescale_acc<D>(tO, alpha);
  const float2 cc = make_float2(c, c);
  const float2 mc = make_float2(-m * c, -m * c);
#pragma unroll
  for (int base = 0; base < kWidth; base += kPart) {
    uint32_t r[kPart];
#pragma unroll
    for (int b = 0; b < kPart; b += 32) tmem_ld32(tS + base + b, *reinterpret_cast<uint32_t(*)[32]>(r + b));
    tmem_wait_ld();
    if (valid < base + kPart) {
#pragma unroll
      for (int i = 0; i < kPart; ++i)
        if (base + i >= valid) r[i] = __float_as_uint(-INFINITY);
    }
#pragma unroll
    for (int i = 0; i < kPart / 2; ++i) {
      const float2 x = fma2(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), cc, mc);
      r[i] = pack_bf16x2(ex2(x.x), ex2(x.y));
    }
    if (kPart == 64) tmem_st32(tP + base / 2, *reinterpret_cast<uint32_t(*)[32]>(r));
    else tmem_st16(tP + base / 2, *reinterpret_cast<uint32_t(*)[16]>(r));
  }
  tmem_wait_st();
}

// ------------------------------------------------------------ split kernel
struct SplitParams {
  int N, M, H, qtiles, splits, split_len;
  float* part_z;            // [BH][qtiles][splits][128][D]
  float* part_l;            // [BH][qtiles][splits][128]
  unsigned* counters;       // [BH][qgroups]
  const __nv_bfloat16* qf;  // synthesis: [H][M][D]
  const float* gate;        // synthesis: [H]
  __nv_bfloat16* out;       // synthesis: Q; encode: Z ([BH][M][D])
  float* dbg_a;             // synthesis: Qd; encode: Z (as rounded)
  float* dbg_b;             // synthesis: Q (as rounded); encode: L
};

struct SlotPlan {
  int mode;
  int qt[2];     // latent block of each slot
  int steps[2];  // steps each slot processes
};

__device__ __forceinline__ SlotPlan slot_plan(int M, int qtiles, int group, int T) {
  SlotPlan s;
  if (M <= 64) {
    s.mode = kLanes;
    s.qt[0] = s.qt[1] = 0;
  } else if (2 * group + 1 < qtiles) {
    s.mode = kPair;
    s.qt[0] = 2 * group;
    s.qt[1] = 2 * group + 1;
  } else {
    s.mode = kStreams;
    s.qt[0] = s.qt[1] = 2 * group;
  }
  for (int k = 0; k < 2; ++k) {
    if (s.mode == kLanes) s.steps[k] = T > 2 * k ? (T - 2 * k + 3) / 4 : 0;
    else if (s.mode == kStreams) s.steps[k] = T > k ? (T - k + 1) / 2 : 0;
    else s.steps[k] = T;
  }
  return s;
}

// Token tile of slot k at step j (in the lanes mode lanes 64-127 take tile + 1).
__device__ __forceinline__ int slot_tile(const SlotPlan& s, int k, int j) {
  if (s.mode == kLanes) return 4 * j + 2 * k;
  if (s.mode == kStreams) return 2 * j + k;
  return j;
}

template <int D, bool kSynth>
__global__ void __launch_bounds__(kThreads, 1)
    split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const SplitParams p) {
  using L = Layout<D>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ Shared sh;
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  constexpr uint32_t kStageBytes = kSynth ? L::kTileBytes : 2 * L::kTileBytes;
  unsigned char* sQ = smem;                                   // [2][128][D]
  unsigned char* sStage = smem + 2 * L::kTileBytes;           // [kStages] x (K, V)
  unsigned char* sOnes = sStage + kStages * kStageBytes;      // [128][D] rows [1, 0, ...]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x, group = blockIdx.y, bh = blockIdx.z;
  const int h = bh % p.H;
  const int n_begin = split * p.split_len;
  const int n_end = min(p.N, n_begin + p.split_len);
  const int T = n_begin < n_end ? (n_end - n_begin + kTile - 1) / kTile : 0;
  const SlotPlan sp = slot_plan(p.M, p.qtiles, group, T);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
      mbar_init(&sh.norm[s], 64);
    }
    mbar_init(&sh.q_full, 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&sh.s_full[k], 1);
      mbar_init(&sh.p_full[k], 128);
      mbar_init(&sh.o_full[k], 1);
    }
    mbar_init(&sh.drain, 1);
    sh.abort = 0;
    sh.last = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 4) fill_ones<D>(sOnes, threadIdx.x - 128, 256);
  fence_proxy_async_smem();
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
      mbar_arrive_expect_tx(&sh.q_full, (sp.mode == kPair ? 2 : 1) * L::kTileBytes);
      if (sp.mode == kLanes) {
        // the 64 (or fewer) latents twice: lanes 64-127 repeat lanes 0-63
        tma_load_3d(sQ, &tm_q, &sh.q_full, 0, 0, qz);
        tma_load_3d(sQ + L::kTileBytes / 2, &tm_q, &sh.q_full, 0, 0, qz);
      } else {
        tma_load_3d(sQ, &tm_q, &sh.q_full, 0, sp.qt[0] * kTile, qz);
        if (sp.mode == kPair) tma_load_3d(sQ + L::kTileBytes, &tm_q, &sh.q_full, 0, sp.qt[1] * kTile, qz);
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
        mbar_wait(&sh.q_full, 0, kWaitLimit);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t aQ0 = smem_u32(sQ);
      const uint32_t aQ1 = sp.mode == kPair ? aQ0 + L::kTileBytes : aQ0;
      const uint32_t aOnes = smem_u32(sOnes);
      const uint32_t idS = idesc_bf16(128, kTile, false, false);
      const uint32_t idO = idesc_bf16(128, L::kNo, false, true);
      constexpr uint32_t kLo = 0u, kAll = 0xFFFFFFFFu;
      auto stage_addr = [&](int t) { return smem_u32(sStage + (t % kStages) * kStageBytes); };
      auto ready = [&](int t) -> bool {
        return wait_or_abort(sh, kSynth ? &sh.norm[t % kStages] : &sh.full[t % kStages], (t / kStages) & 1);
      };
      // scores of slot k, step j
      auto issue_s = [&](int k, int j) -> bool {
        const uint32_t dS = tmem + k * kSlotCols;
        const uint32_t aQ = k == 0 ? aQ0 : aQ1;
        const int t = slot_tile(sp, k, j);
        if (!ready(t)) return false;
        if (sp.mode == kLanes) {
          const bool has_b = t + 1 < T;
          if (has_b && !ready(t + 1)) return false;
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < D / 16; ++q)
            mma_ss_masked(dS, L::kmajor(aQ, q), L::kmajor(stage_addr(t), q), idS, q > 0, kLo, kLo, kAll, kAll);
          if (has_b) {
#pragma unroll
            for (int q = 0; q < D / 16; ++q)
              mma_ss_masked(dS, L::kmajor(aQ, q), L::kmajor(stage_addr(t + 1), q), idS, q > 0, kAll, kAll, kLo,
                            kLo);
          }
        } else {
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < D / 16; ++q) mma_ss(dS, L::kmajor(aQ, q), L::kmajor(stage_addr(t), q), idS, q > 0);
        }
        mma_commit(&sh.s_full[k]);
        return true;
      };
      // O += P [V | 1] for slot k, step j; releases the tiles no longer needed
      auto issue_pv = [&](int k, int j) {
        const uint32_t dO = tmem + k * kSlotCols + kColO;
        const uint32_t aP = tmem + k * kSlotCols + kColP;
        const int t = slot_tile(sp, k, j);
        const uint32_t vA = stage_addr(t) + (kSynth ? 0 : L::kTileBytes);
        if (sp.mode == kLanes) {
          const bool has_b = t + 1 < T;
          const uint32_t vB = stage_addr(t + 1) + (kSynth ? 0 : L::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts_masked(dO, aP + kk * 8, L::values1(vA, aOnes, kk), idO, (j > 0 || kk > 0), kLo, kLo, kAll, kAll);
          if (has_b) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ts_masked(dO, aP + kk * 8, L::values1(vB, aOnes, kk), idO, (j > 0 || kk > 0), kAll, kAll, kLo,
                            kLo);
          }
          mma_commit(&sh.empty[t % kStages]);
          if (has_b) mma_commit(&sh.empty[(t + 1) % kStages]);
        } else {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts(dO, aP + kk * 8, L::values1(vA, aOnes, kk), idO, (j > 0 || kk > 0));
          if (sp.mode == kStreams || k == 1) mma_commit(&sh.empty[t % kStages]);
        }
      };
      bool ok = wait_or_abort(sh, &sh.q_full, 0);
      for (int k = 0; ok && k < 2; ++k)
        if (sp.steps[k] > 0) ok = issue_s(k, 0);
      const int jmax = max(sp.steps[0], sp.steps[1]);
      for (int j = 0; ok && j < jmax; ++j) {
        for (int k = 0; ok && k < 2; ++k) {
          if (j >= sp.steps[k]) continue;
          if (!wait_or_abort(sh, &sh.p_full[k], j & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(k, j);
          if (j + 1 < sp.steps[k]) ok = issue_s(k, j + 1);
        }
      }
      mma_commit(&sh.o_full[0]);
      mma_commit(&sh.o_full[1]);
      // every MMA of this CTA completes before TMEM is released
      mma_commit(&sh.drain);
      mbar_wait(&sh.drain, 0, kWaitLimit);
    }
  } else if (warp < 4) {
    // ------------------------------------------- N0 of the synthesis tiles
    if (kSynth) {
      const int nt = threadIdx.x - 64;  // 0..63: rows nt and nt + 64 of each tile
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
            for (int q = 0; q < 4; ++q) {
              const float a = __uint_as_float(w[q] << 16), b = __uint_as_float(w[q] & 0xFFFF0000u);
              ss = fmaf(a, a, fmaf(b, b, ss));
            }
          }
          const float r = rsqrtf(ss / (float)D + kEps);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) {
            uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
              w[q] = pack_bf16x2(__uint_as_float(w[q] << 16) * r, __uint_as_float(w[q] & 0xFFFF0000u) * r);
            row[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&sh.norm[s]);
      }
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int k = (warp - 4) >> 2;  // slot
    const int row = (threadIdx.x - 128) & 127;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + k * kSlotCols;
    const uint32_t tO = tS + kColO;
    const int half = sp.mode == kLanes ? (row >> 6) : 0;
    const int r_in = sp.mode == kLanes ? (row & 63) : row;
    const int qt = sp.qt[k];
    const int latent = qt * kTile + r_in;
    const bool valid = latent < p.M;
    const float c = rsqrtf((float)D) * kLog2e;
    float m = -INFINITY;
    bool has_acc = false;
    bool ok = true;
    for (int j = 0; j < sp.steps[k]; ++j) {
      if (!wait_or_abort(sh, &sh.s_full[k], j & 1)) { ok = false; break; }
      tc_fence_after();
      const int t = slot_tile(sp, k, j) + half;
      if (t < T) {
        const int n0 = n_begin + t * kTile;
        softmax_step<D, kTile>(tS, tS + kColP, tO, min(kTile, n_end - n0), c, m, has_acc);
        has_acc = true;
      }
      tc_fence_before();
      mbar_arrive(&sh.p_full[k]);
    }
    // both slots' products are complete before the stage buffers are reused
    // as scratch below
    if (ok) ok = wait_or_abort(sh, &sh.o_full[k], 0);
    if (ok) ok = wait_or_abort(sh, &sh.o_full[k ^ 1], 0);
    tc_fence_after();
    float o[D];
    const float l = load_acc<D>(tO, o);
    (void)valid;

    // 1) each token stream's (L, Z) into shared memory
    constexpr int kZs = D + 1;  // padded row stride
    float* scr_l = reinterpret_cast<float*>(sStage);  // [256]
    float* scr_z = scr_l + 256;                       // [256][D + 1]
    const int e = threadIdx.x - 128;
    {
      const bool any = ok && has_acc && l > 0.f;  // a stream with no token never wrote its accumulator
      const float inv = any ? 1.f / l : 0.f;
      scr_l[e] = any ? (m * c + __log2f(l)) * kLn2 : -INFINITY;
#pragma unroll
      for (int d = 0; d < D; ++d) scr_z[e * kZs + d] = any ? o[d] * inv : 0.f;
    }
    softmax_groups_sync();

    // 2) one partial result per (latent row, split): the CTA's token streams of
    //    a row merged first (Appendix B.3 schedule over the streams)
    {
      int nent = 1, stride = 0, r_w = row, qt_w = sp.qt[k];
      bool writer = true;
      if (sp.mode == kLanes) {
        writer = e < 64; nent = 4; stride = 64; r_w = e; qt_w = sp.qt[0];
      } else if (sp.mode == kStreams) {
        writer = e < 128; nent = 2; stride = 128; r_w = e; qt_w = sp.qt[0];
      }
      const int latent_w = qt_w * kTile + r_w;
      if (writer && latent_w < p.M) {
        float lmax = -INFINITY;
        for (int i = 0; i < nent; ++i) lmax = fmaxf(lmax, scr_l[e + i * stride]);
        float u[D], dsum = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) u[d] = 0.f;
        for (int i = 0; i < nent; ++i) {
          const float li = scr_l[e + i * stride];
          const float w = li == -INFINITY ? 0.f : __expf(li - lmax);
          dsum += w;
#pragma unroll
          for (int d = 0; d < D; ++d) u[d] = fmaf(w, scr_z[(e + i * stride) * kZs + d], u[d]);
        }
        const float invd = dsum > 0.f ? 1.f / dsum : 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) u[d] *= invd;
        const size_t prow = (((size_t)bh * p.qtiles + qt_w) * p.splits + split) * kTile + r_w;
        store_row<D>(p.part_z + prow * D, u);
        p.part_l[prow] = dsum > 0.f ? lmax + __logf(dsum) : -INFINITY;
      }
    }
    __threadfence();
    softmax_groups_sync();
    const size_t grp = (size_t)bh * gridDim.y + group;
    if (threadIdx.x == 128) {
      const unsigned prev = atomicAdd(p.counters + grp, 1u);
      sh.last = prev == (unsigned)(p.splits - 1);
    }
    softmax_groups_sync();
    if (sh.last) {
      __threadfence();
      if (threadIdx.x == 128) p.counters[grp] = 0u;  // ready for the next call
      // 3) the last CTA of the group merges the splits (Appendix B.3:
      //    L_max, d_s = exp(L_s - L_max), U = sum d_s Z_s, Z = U / d), with
      //    `tpr` threads per latent row sharing the splits
      const int rows = sp.mode == kLanes ? 64 : (sp.mode == kStreams ? 128 : 256);
      const int tpr = 256 / rows;
      const int rg = e / tpr, part = e % tpr;
      const int qt_f = sp.mode == kPair ? sp.qt[rg >> 7] : sp.qt[0];
      const int r_f = rg & 127;
      const int latent_f = qt_f * kTile + r_f;
      const size_t base = ((size_t)bh * p.qtiles + qt_f) * p.splits * kTile + r_f;
      float lmax = -INFINITY;
#pragma unroll 4
      for (int sidx = part; sidx < p.splits; sidx += tpr)
        lmax = fmaxf(lmax, __ldcg(p.part_l + base + (size_t)sidx * kTile));
      float u[D], dsum = 0.f;
#pragma unroll
      for (int d = 0; d < D; ++d) u[d] = 0.f;
#pragma unroll 2
      for (int sidx = part; sidx < p.splits; sidx += tpr) {
        const size_t r = base + (size_t)sidx * kTile;
        const float ls = __ldcg(p.part_l + r);
        const float w = ls == -INFINITY ? 0.f : __expf(ls - lmax);
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
      // combine the tpr threads of a row (consecutive lanes of one warp)
      float gmax = lmax;
      for (int off = 1; off < tpr; off <<= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xFFFFFFFFu, gmax, off));
      const float sc = lmax == -INFINITY ? 0.f : __expf(lmax - gmax);
      dsum *= sc;
#pragma unroll
      for (int d = 0; d < D; ++d) u[d] *= sc;
      for (int off = 1; off < tpr; off <<= 1) {
        dsum += __shfl_xor_sync(0xFFFFFFFFu, dsum, off);
#pragma unroll
        for (int d = 0; d < D; ++d) u[d] += __shfl_xor_sync(0xFFFFFFFFu, u[d], off);
      }
      if (part == 0 && latent_f < p.M) {
        const float invd = 1.f / dsum;
#pragma unroll
        for (int d = 0; d < D; ++d) u[d] *= invd;
        const size_t orow = (size_t)bh * p.M + latent_f;
        if (kSynth) {
          // gate (eq. 7): Q = N0(Qf) + g * Qd in fp32, cast to bf16
          float f[D];
          load_row<D>(p.qf + ((size_t)h * p.M + latent_f) * D, f);
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
          if (p.dbg_b) p.dbg_b[orow] = gmax + __logf(dsum);
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
__global__ void __launch_bounds__(kThreads, 1)
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
  unsigned char* sOnes = sK + kStages * L::kTileBytes;     // [128][D]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int n_tiles = (p.N + kTile - 1) / kTile;
  const int t_begin = blockIdx.x * p.tiles_per_cta;
  const int T = max(0, min(n_tiles, t_begin + p.tiles_per_cta) - t_begin);
  // slot k takes local tiles k, k+2, ...; each tile runs `chunks` route blocks
  int steps[2];
  for (int k = 0; k < 2; ++k) steps[k] = T > k ? ((T - k + 1) / 2) * chunks : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    mbar_init(&sh.q_full, 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&sh.s_full[k], 1);
      mbar_init(&sh.p_full[k], 128);
      mbar_init(&sh.o_full[k], 1);
    }
    mbar_init(&sh.drain, 1);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 4) fill_ones<D>(sOnes, threadIdx.x - 128, 256);
  fence_proxy_async_smem();
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
      const uint32_t aQ = smem_u32(sQ), aZ = smem_u32(sZ), aOnes = smem_u32(sOnes);
      const uint32_t idO = idesc_bf16(128, L::kNo, false, true);
      // step u of slot k: local tile k + 2*(u / chunks), route block u % chunks
      auto issue_s = [&](int k, int u) -> bool {
        const int t = k + 2 * (u / chunks), ch = u % chunks;
        const int s = t % kStages;
        if (ch == 0) {
          if (!wait_or_abort(sh, &sh.full[s], (t / kStages) & 1)) return false;
          tc_fence_after();
        }
        const int width = min(kTile, p.M - ch * kTile);
        const uint32_t aK = smem_u32(sK + s * L::kTileBytes);
#pragma unroll
        for (int q = 0; q < D / 16; ++q)
          mma_ss(tmem + k * kSlotCols, L::kmajor(aK, q), L::kmajor(aQ + ch * L::kTileBytes, q),
                 idesc_bf16(128, width, false, false), q > 0);
        if (ch == chunks - 1) mma_commit(&sh.empty[s]);
        mma_commit(&sh.s_full[k]);
        return true;
      };
      auto issue_pv = [&](int k, int u) {
        const int ch = u % chunks;
        const int width = min(kTile, p.M - ch * kTile);
        const uint32_t zc = aZ + ch * L::kTileBytes;
        for (int kk = 0; kk < width / 16; ++kk)
          mma_ts(tmem + k * kSlotCols + kColO, tmem + k * kSlotCols + kColP + kk * 8, L::values1(zc, aOnes, kk), idO,
                 (ch > 0 || kk > 0));
        if (ch == chunks - 1) mma_commit(&sh.o_full[k]);
      };
      bool ok = wait_or_abort(sh, &sh.q_full, 0);
      for (int k = 0; ok && k < 2; ++k)
        if (steps[k] > 0) ok = issue_s(k, 0);
      const int umax = max(steps[0], steps[1]);
      for (int u = 0; ok && u < umax; ++u) {
        for (int k = 0; ok && k < 2; ++k) {
          if (u >= steps[k]) continue;
          if (!wait_or_abort(sh, &sh.p_full[k], u & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(k, u);
          if (u + 1 < steps[k]) ok = issue_s(k, u + 1);
        }
      }
      mma_commit(&sh.drain);
      mbar_wait(&sh.drain, 0, kWaitLimit);
    }
  } else if (warp >= 4) {
    const int k = (warp - 4) >> 2;
    const int row = (threadIdx.x - 128) & 127;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + k * kSlotCols;
    const uint32_t tO = tS + kColO;
    const float c = rsqrtf((float)D) * kLog2e;
    float m = -INFINITY;
    for (int u = 0; u < steps[k]; ++u) {
      const int ch = u % chunks;
      if (!wait_or_abort(sh, &sh.s_full[k], u & 1)) break;
      tc_fence_after();
      if (ch == 0) m = -INFINITY;
      const int width = min(kTile, p.M - ch * kTile);
      if (width > 64) softmax_step<D, kTile>(tS, tS + kColP, tO, width, c, m, ch > 0);
      else if (width > 32) softmax_step<D, 64>(tS, tS + kColP, tO, width, c, m, ch > 0);
      else softmax_step<D, 32>(tS, tS + kColP, tO, width, c, m, ch > 0);
      tc_fence_before();
      mbar_arrive(&sh.p_full[k]);
      if (ch == chunks - 1) {
        const int t = k + 2 * (u / chunks);
        if (!wait_or_abort(sh, &sh.o_full[k], (u / chunks) & 1)) break;
        tc_fence_after();
        float y[D];
        const float l = load_acc<D>(tO, y);
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
  return 1024 + 3 * (size_t)Layout<D>::kTileBytes + kStages * stage;
}

template <int D>
size_t decode_smem(int M) {
  const int chunks = (M + kTile - 1) / kTile;
  return 1024 + (2 * chunks + kStages + 1) * (size_t)Layout<D>::kTileBytes;
}

template <int D>
cudaError_t forward_d(const DeviceProblem& pr, const TcPlan& pl, const TcWorkspace& ws, cudaEvent_t* ev,
                      cudaStream_t stream, const char** failed) {
  const int BH = pr.B * pr.H;
  cudaError_t e;
  CUtensorMap m_seed, m_ks, m_qbuf, m_k, m_v, m_qdec, m_zdec;
  const int qbox = pr.M <= 64 ? 64 : kTile;
  *failed = "cuTensorMapEncodeTiled";
  if (!make_map(&m_seed, pr.Qseed, D, pr.M, pr.H, qbox) || !make_map(&m_ks, pr.Ks, D, pr.N, BH, kTile) ||
      !make_map(&m_qbuf, ws.q, D, pr.M, BH, qbox) || !make_map(&m_k, pr.K, D, pr.N, BH, kTile) ||
      !make_map(&m_v, pr.V, D, pr.N, BH, kTile) || !make_map(&m_qdec, ws.q, D, pr.M, BH, kTile) ||
      !make_map(&m_zdec, ws.z, D, pr.M, BH, kTile))
    return cudaErrorInvalidValue;

  const dim3 grid(pl.splits, pl.qgroups, BH);
  SplitParams sp{};
  sp.N = pr.N; sp.M = pr.M; sp.H = pr.H;
  sp.qtiles = pl.tiles; sp.splits = pl.splits; sp.split_len = pl.split_len;
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
    a.counters = ws.counters + (size_t)BH * pl.qgroups;
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

// The split count (per latent group) with the least estimated time when each
// CTA holds one SM: waves x (per-CTA overhead + token tiles per CTA), the
// overhead counted in token tiles (set-up, pipeline fill, partial results and
// merge). Fewer splits win ties.
int choose_splits(long long groups, int n_tiles, int sms, int min_tiles, int overhead_tiles, int forced) {
  if (forced > 0) return std::min(forced, std::max(1, n_tiles));
  const int max_splits = std::max(1, n_tiles / std::max(1, min_tiles));
  int best = 1;
  double best_cost = 1e300;
  for (int s = 1; s <= std::min(max_splits, 2048); ++s) {
    const int per = (n_tiles + s - 1) / s;
    const int real = (n_tiles + per - 1) / per;
    const long long waves = (groups * real + sms - 1) / sms;
    const double cost = (double)waves * (overhead_tiles + per);
    if (cost < best_cost * 0.99) {
      best_cost = cost;
      best = real;
    }
  }
  return best;
}

}  // namespace tc

TcPlan tc_plan(int B, int H, int N, int M, int D, int sms, int forced_splits) {
  (void)D;
  TcPlan pl{};
  const long long BH = (long long)B * H;
  const int n_tiles = (N + tc::kTile - 1) / tc::kTile;
  pl.tiles = M <= 64 ? 1 : (M + tc::kTile - 1) / tc::kTile;
  pl.qgroups = M <= 128 ? 1 : (pl.tiles + 1) / 2;
  pl.streams = 1;  // the token streams of a CTA are merged before its partial is written
  // token tiles per split: at least 4 (two per slot) when the sequence allows
  const int splits = tc::choose_splits(BH * pl.qgroups, n_tiles, std::max(1, sms), 4, 8, forced_splits);
  const int tiles_per_split = (n_tiles + splits - 1) / splits;
  pl.split_len = tiles_per_split * tc::kTile;
  pl.splits = (N + pl.split_len - 1) / pl.split_len;
  // decode: one CTA per SM over consecutive token tiles of one head
  const int dsplit = tc::choose_splits(BH, n_tiles, std::max(1, sms), 2, 4, 0);
  const int per = (n_tiles + dsplit - 1) / dsplit;
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
