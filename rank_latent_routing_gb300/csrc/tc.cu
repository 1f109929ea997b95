// Tensor-core (tcgen05 + TMEM + TMA) kernels of the FLARE++ mixer forward,
// bf16 inputs, fp32 softmax and accumulation.
//
// Two kernels carry the three attention calls of the mixer (FLARE++ paper,
// Section 3.2 eq. 6 and eq. 8):
//
//  * split_kernel — latent queries attend over one token range (split) of a
//    head. Scores S = Q K^T land in TMEM; threads run an online softmax over
//    the tokens; P goes back to TMEM in bf16 over the scores and the tensor
//    core accumulates O += P [V | 1] in TMEM, the appended ones column giving
//    the softmax row sum. Each split's (Z_s, L_s) goes to global memory and
//    the last CTA of a head to arrive merges all splits with the stable
//    log-sum-exp schedule of Appendix B.3 (eq. 29-33). The synthesis instance
//    normalises each staged Ks_raw tile in place (N0, eq. 5), uses it as both
//    keys and values (eq. 19) and ends with the gate (eq. 7):
//    Q = N0(Qf) + g * Qd in fp32, cast to bf16. The encode instance ends with
//    Z (bf16) and L.
//  * decode_kernel — tokens attend over the M routes: Q and Z of the head stay
//    in shared memory for all of the CTA's token tiles; each column half of a
//    TMEM slot owns a token tile and computes S = K Q^T 64 routes at a time
//    with an online softmax over M per token, and O += P [Z | 1];
//    out = O / rowsum in bf16.
//
// One CTA per SM, 512 threads: warp 0 issues TMA loads, warps 1-4 issue the
// MMAs (one thread each, one per (slot, column half); warp 1 owns TMEM),
// warps 0, 5, 14 and 15 (one per SM sub-partition) normalise a quarter of
// every synthesis tile each, and two softmax warpgroups (warps 6-9 and
// 10-13) take the first and the second 64 score columns of every step.
// Both work on two TMEM slots in turn, so the tensor core computes one slot's
// products and next scores while the softmax runs on the other. Each (slot,
// half) is a pipeline of its own: its issuing thread adds the half's products
// and then writes the half's next 64 score columns, and its warpgroup waits
// for those alone. A thread spends ~50-80 cycles issuing one tcgen05.mma, so
// four issuers keep the tensor pipe fed where one or two would not. Warp w
// reads TMEM lanes 32*(w%4) .. +31.
//
// A slot holds 128 score columns and two accumulators, one per column half:
// each half writes its P in bf16 over the first 32 of its own score columns,
// and its products go to its own accumulator, so the two halves of a row are
// two independent softmax streams (own reference, own accumulator) that meet
// only at the end, in the same log-sum-exp merge as the splits. The next
// scores are issued after the products that read P; the tensor core runs a
// thread's MMAs in order.
//
// The softmax is one pass: p = 2^(s*c - r) against a reference r (an integer
// in exp2 units) fixed before the tile; the first tile of a stream sets r
// from its own max. Whether some p reached 2 is read off the packed bf16
// results (exponent field >= 128 <=> p >= 2, which also catches inf); only
// then does the warp read its scores again, move r to 16 units above the
// ceiling of their max and redo them, and the accumulator is rescaled
// exactly by 2^(r_old - r_new) before the tile's products are added.
//
// Every wait on an mbarrier is bounded: after about a second without progress
// the thread records kErrTimeout in the device error word, raises the CTA's
// abort flag and leaves its loop, so a broken invariant ends the kernel
// instead of hanging the GPU.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"
#include "tmap.h"

namespace flarepp {
namespace tc {

using namespace sm100;

__device__ unsigned g_tc_error = 0u;

#ifdef FLAREPP_TRACE
// Pipeline trace (trace builds only): clock64 stamps of block 0 of one pass,
// g_trace[role][i]. g_trace_pass picks the pass: 1 synthesis, 2 encode (and
// the simplified synthesis), 3 decode; 0 records nothing.
constexpr int kTraceRoles = 16, kTraceLen = 4096;
__device__ unsigned long long g_trace[kTraceRoles][kTraceLen];
__device__ int g_trace_pass = 0;
// roles: kernel start/end; TMA issue per tile; N0 per tile (4 parts);
// issuing threads (slot, half) per step; softmax warps of the two halves
// per (step, slot); epilogue phases
enum : int { kTrStart = 0, kTrLoad = 1, kTrNorm = 2, kTrIssue = 6, kTrSoftmax = 10, kTrEpi = 12 };
__device__ __forceinline__ void trace_stamp(bool on, int role, int i) {
  if (on && i >= 0 && i < kTraceLen) g_trace[role][i] = clock64();
}
#define FLAREPP_TR(on, role, i) trace_stamp((on), (role), (i))
#else
#define FLAREPP_TR(on, role, i) ((void)0)
#endif

constexpr int kThreads = 512;
constexpr int kWarpIssue = 1;        // first MMA-issuing warp: warp 1 + 2k + hf
constexpr int kWarpNorm = 5;         // N0 of the synthesis tiles: warps 0, 5, 14 and 15
constexpr int kWarpSoftmax = 6;      // first softmax warp (6-13)
constexpr int kTile = 128;           // tokens per staged tile; latents per row block
constexpr int kMaxStages = 16;       // token-tile ring depth (upper bound)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSlotCols = 256;  // slot s starts at column 256*s
constexpr uint32_t kColO = 128;      // accumulator of column half 0; half 1's follows it
constexpr uint32_t kColQ = 224;      // the slot's latent queries (bf16 pairs), A operand of the scores
constexpr long long kWaitLimit = 2000000000LL;  // clock cycles (~1 s)
// under the test hook that makes one barrier never complete, waits give up
// after ~1 ms, so that the forced timeout ends the call quickly
constexpr long long kTestWaitLimit = 2000000LL;

// How the two TMEM slots of a split-kernel CTA divide the work:
//  kLanes   (M <= 64)  each slot holds the latents twice; lanes 0-63 and 64-127
//                      score different token tiles (4 token streams per CTA);
//  kStreams            one 128-row latent block, the slots take alternate tiles;
//  kPair               two 128-row latent blocks, both slots see every tile.
enum : int { kLanes = 0, kStreams = 1, kPair = 2 };

struct Shared {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t norm[kMaxStages];
  uint64_t q_full;
  uint64_t s_full[2][2];  // scores of half h of slot k ready (and the half's earlier products done)
  uint64_t p_full[2][2];  // P of column half h of slot k written
  uint64_t o_full[2][2];  // the last products of half h of slot k done
  uint64_t q_tmem;        // the latent queries are in TMEM
  uint64_t drain;         // every MMA of the CTA has completed
  long long wait_limit;   // clock cycles a wait may take before it gives up
  uint32_t tmem_base;
  int abort;
  int last;
};

// A phase that has completed is taken at once; the abort flag is read only on
// the slow path, so a wait that needs no waiting costs no shared-memory load.
// kSleep: the thread sleeps in the barrier between tests (for long,
// latency-tolerant waits: a producer a ring ahead) instead of polling, which
// would take issue slots from the warps beside it.
template <bool kSleep = false>
__device__ __forceinline__ bool wait_or_abort(Shared& sh, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*(volatile int*)&sh.abort) return false;
  if (kSleep ? mbar_wait_sleep(bar, parity, sh.wait_limit) : mbar_wait(bar, parity, sh.wait_limit)) return true;
  atomicOr(&g_tc_error, kErrTimeout);
  *(volatile int*)&sh.abort = 1;
  return false;
}

// wait_or_abort by every lane of a convergent warp; the warp agrees on the
// outcome (a lane that gave up makes the whole warp give up), so that the
// warp stays convergent for the elect.sync-issued MMAs that follow.
__device__ __forceinline__ bool warp_wait(Shared& sh, uint64_t* bar, uint32_t parity) {
  const bool ok = wait_or_abort(sh, bar, parity);
  return __all_sync(0xFFFFFFFFu, ok);
}

// One arrival per warp: the lanes' TMEM accesses are ordered before the
// warp's sync, then lane 0 arrives.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Barrier over the two softmax warpgroups only (256 threads).
__device__ __forceinline__ void softmax_groups_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// 2^e for an integer e <= 0 held in a float (exact; 0 below the normal range).
__device__ __forceinline__ float pow2_neg(float e) {
  return e < -126.f ? 0.f : __int_as_float((127 + static_cast<int>(e)) << 23);
}

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
  // A descriptor moved `bytes` further (the start field holds address / 16;
  // shared-memory addresses stay below 2^18, so no carry leaves the field).
  static __device__ __forceinline__ uint64_t adv(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }
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

// Scales this lane's accumulator (values and row sum) by `alpha`.
template <int D>
__device__ __forceinline__ void rescale_acc(uint32_t tO, float alpha) {
  uint32_t r[16];
#pragma unroll
  for (int c = 0; c < Layout<D>::kNo; c += 16) {
    tmem_ld16(tO + c, r);
    tmem_wait_ld_regs(r);
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
    tmem_st16(tO + c, r);
  }
  tmem_wait_st();
}

// Reads the D output values and the row sum of this lane's accumulator.
template <int D>
__device__ __forceinline__ float load_acc(uint32_t tO, float (&o)[D]) {
  uint32_t a[32];
  tmem_ld32(tO, a);
  if (D == 32) {
    uint32_t s[16];
    tmem_ld16(tO + 32, s);
    tmem_wait_ld_regs(a);
    tmem_wait_ld_regs(s);
#pragma unroll
    for (int i = 0; i < D; ++i) o[i] = __uint_as_float(a[i]);
    return __uint_as_float(s[0]);
  }
  tmem_wait_ld_regs(a);
#pragma unroll
  for (int i = 0; i < D; ++i) o[i] = __uint_as_float(a[i]);
  return __uint_as_float(a[D]);
}

// ------------------------------------------------------------- softmax step
// Reads this lane's 64 scores of a column half and masks the columns at or
// past `valid` (1..64).
__device__ __forceinline__ void load_half(uint32_t tS, int valid, uint32_t (&s)[64]) {
  tmem_ld64(tS, s);
  tmem_wait_ld_regs(s);
  if (valid < 64) {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (i >= valid) s[i] = __float_as_uint(-INFINITY);
  }
}

// p = 2^(s*c - r) of the 64 columns, packed in bf16 pairs into s[0..31];
// returns the OR of the packed words.
__device__ __forceinline__ uint32_t exp_pack(uint32_t (&s)[64], float c, float r) {
  const float2 cc = make_float2(c, c);
  const float2 rr = make_float2(-r, -r);
  uint32_t o0 = 0u, o1 = 0u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float2 x = fma2(make_float2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), cc, rr);
    s[i] = pack_bf16x2(ex2(x.x), ex2(x.y));
    if (i & 1) o1 |= s[i];
    else o0 |= s[i];
  }
  return o0 | o1;
}

// Exponent field >= 128 in either bf16 half: some p >= 2 (or inf / NaN).
constexpr uint32_t kGrowBits = 0x40004000u;
// When the reference moves it is set this many exp2 units above the tile max,
// so that p <= 2^-16 and the next move waits for the max to grow by 17 units
// (p that small loses nothing: fp32 and bf16 keep their relative precision
// down to 2^-126).
constexpr float kHeadroom = 16.0f;

__device__ __forceinline__ float half_max(const uint32_t (&s)[64]) {
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int i = 0; i < 64; i += 4) {
    m0 = max3(m0, __uint_as_float(s[i]), __uint_as_float(s[i + 1]));
    m1 = max3(m1, __uint_as_float(s[i + 2]), __uint_as_float(s[i + 3]));
  }
  return fmaxf(m0, m1);
}

// One softmax step of this lane over its column half at tS: `valid` (<= 64)
// columns, P (32 packed columns) written over the first 32. The first tile
// of a stream (r = -inf, the same for the whole warp) takes its reference
// from its own max; later tiles are done against r in one pass, and only if
// some p reached 2 is the half read again and redone against a new r.
// Warp-uniform `valid`.
__device__ __forceinline__ void softmax_half(uint32_t tS, int valid, float c, float& r) {
  uint32_t s[64];
  load_half(tS, valid, s);
  if (__any_sync(0xFFFFFFFFu, r == -INFINITY)) {
    const float m = half_max(s);
    if (r == -INFINITY) r = ceilf(m * c) + kHeadroom;
    exp_pack(s, c, r);
  } else {
    const uint32_t bits = exp_pack(s, c, r);
    if (__any_sync(0xFFFFFFFFu, (bits & kGrowBits) != 0u)) {
      // the scores are still in TMEM
      load_half(tS, valid, s);
      const float m = half_max(s);
      if ((bits & kGrowBits) != 0u) r = ceilf(m * c) + kHeadroom;
      exp_pack(s, c, r);
    }
  }
  tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(s));
}

// End of a softmax step: the products of the previous step are in (this
// step's scores were issued after them), so the accumulator is brought to the
// reference of the probabilities just written; then P goes to the tensor core.
template <int D>
__device__ __forceinline__ void finish_half(uint64_t* p_full, uint32_t tO, float r, float& ro, bool acc) {
  tmem_wait_st();
  const bool need = acc && ro != r;
  if (__any_sync(0xFFFFFFFFu, need)) rescale_acc<D>(tO, need ? pow2_neg(ro - r) : 1.f);
  ro = r;
  warp_arrive(p_full);
}

// N0 (eq. 5) of rows 32*part + lane of staged synthesis tile t, in place, in
// the swizzled layout (a row's 16-byte chunks are permuted within the row,
// which the sum of squares and the scaling do not see); one arrival per warp
// on the tile's barrier. Returns false if the wait for the tile gave up.
template <int D, int kStages>
__device__ __forceinline__ bool normalise_part(Shared& sh, unsigned char* sStage, uint32_t stage_bytes, int t,
                                               int part, int lane) {
  using L = Layout<D>;
  const int s = t % kStages;
  if (!wait_or_abort(sh, &sh.full[s], (t / kStages) & 1)) return false;
  uint4* row = reinterpret_cast<uint4*>(sStage + s * stage_bytes + (32 * part + lane) * L::kRowBytes);
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
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) mbar_arrive(&sh.norm[s]);
  return true;
}

// ------------------------------------------------------------ split kernel
struct SplitParams {
  int N, M, H, qtiles, splits, split_len;
  float* part_z;            // [BH][qtiles][splits][128][D]
  float* part_l;            // [BH][qtiles][splits][128]
  unsigned* counters;       // [BH][qgroups]
  int q_by_head;            // latent queries [H][M][D] (1) or [BH][M][D] (0)
  const __nv_bfloat16* qf;  // gated passes: [H][M][D]
  const float* gate;        // gated passes: [H]
  __nv_bfloat16* out;       // gated: Q; encode: Z ([BH][M][D])
  float* dbg_a;             // gated: Qd; encode: Z (as rounded)
  float* dbg_b;             // gated: Q (as rounded); encode: L
  int fail_wait;            // test only: P barrier of slot 0, half 0 expects one arrival too many
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

// Epilogue scratch of the split kernel: (L, Z) of 512 softmax streams.
template <int D>
__host__ __device__ constexpr int split_scratch_bytes() {
  return 512 * 4 + 512 * (D + 1) * 4;
}

// Token-tile ring depth of the split kernel: as deep as fits next to the
// latent tiles and the ones tile (within ~200 KB). A stage holds a key tile,
// and a value tile unless the keys serve as values.
template <int D, int kKind>
__host__ __device__ constexpr int split_stages() {
  constexpr int stage = (pass_separate_values(kKind) ? 2 : 1) * Layout<D>::kTileBytes;
  constexpr int n = (200 * 1024 - 3 * Layout<D>::kTileBytes) / stage;
  return n > kMaxStages ? kMaxStages : n;
}

template <int D, int kKind>
__global__ void __launch_bounds__(kThreads, 1)
    split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const SplitParams p) {
  using L = Layout<D>;
  constexpr bool kNormKeys = pass_normalises_keys(kKind);
  constexpr bool kSepValues = pass_separate_values(kKind);
  constexpr int kStages = split_stages<D, kKind>();
  constexpr uint32_t kStageBytes = kSepValues ? 2 * L::kTileBytes : L::kTileBytes;
  constexpr uint32_t kValueOff = kSepValues ? L::kTileBytes : 0;  // value tile within a stage
  static_assert(kStages * (int)kStageBytes >= split_scratch_bytes<D>(), "epilogue scratch exceeds the stage ring");
  extern __shared__ unsigned char smem_raw[];
  __shared__ Shared sh;
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
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
  const int jmax = max(sp.steps[0], sp.steps[1]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], sp.mode == kPair ? 4 : 2);  // one release per issuing thread that reads the tile
      mbar_init(&sh.norm[s], 4);                          // one arrival per normaliser warp
    }
    mbar_init(&sh.q_full, 1);
    for (int k = 0; k < 2; ++k)
      for (int hf = 0; hf < 2; ++hf) {
        mbar_init(&sh.s_full[k][hf], 1);
        // one arrival per softmax warp of the half (one more under the test hook)
        mbar_init(&sh.p_full[k][hf], 4 + (p.fail_wait && k == 0 && hf == 0 ? 1 : 0));
        mbar_init(&sh.o_full[k][hf], 1);
      }
    mbar_init(&sh.drain, 4);
    mbar_init(&sh.q_tmem, 4);
    sh.wait_limit = p.fail_wait ? kTestWaitLimit : kWaitLimit;
    sh.abort = 0;
    sh.last = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= kWarpSoftmax && warp < kWarpSoftmax + 8) fill_ones<D>(sOnes, threadIdx.x - 32 * kWarpSoftmax, 256);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
#ifdef FLAREPP_TRACE
  const bool tr_on = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
                     g_trace_pass == (kKind == kPassEncode ? 2 : 1);
#endif
  FLAREPP_TR(tr_on && threadIdx.x == 0, kTrStart, 0);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // (in the synthesis instance the warp also normalises rows 0-31 of each
    // tile, kStages / 2 tiles behind the loads its lane 0 issues: the load of
    // tile t waits for tile t - kStages to be released, which in the lanes
    // mode needs tile t - kStages + 1 normalised, so the lag must stay below
    // kStages - 1)
    constexpr int kLag = kNormKeys ? kStages / 2 : 0;
    static_assert(kLag <= kStages - 2, "normaliser lag would deadlock the ring");
    int issued = 0;
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      if (kSepValues) prefetch_tmap(&tm_v);
      const int qz = p.q_by_head ? h : bh;
      mbar_arrive_expect_tx(&sh.q_full, (sp.mode == kPair ? 2 : 1) * L::kTileBytes);
      if (sp.mode == kLanes) {
        // the 64 (or fewer) latents twice: lanes 64-127 repeat lanes 0-63
        tma_load_3d(sQ, &tm_q, &sh.q_full, 0, 0, qz);
        tma_load_3d(sQ + L::kTileBytes / 2, &tm_q, &sh.q_full, 0, 0, qz);
      } else {
        tma_load_3d(sQ, &tm_q, &sh.q_full, 0, sp.qt[0] * kTile, qz);
        if (sp.mode == kPair) tma_load_3d(sQ + L::kTileBytes, &tm_q, &sh.q_full, 0, sp.qt[1] * kTile, qz);
      }
    }
    bool ok = true;
    for (int t = 0; t < T + kLag; ++t) {
      if (lane == 0 && ok && t < T) {
        const int s = t % kStages;
        if (t >= kStages && !wait_or_abort<true>(sh, &sh.empty[s], ((t / kStages) - 1) & 1)) {
          ok = false;
        } else {
          unsigned char* dst = sStage + s * kStageBytes;
          mbar_arrive_expect_tx(&sh.full[s], kStageBytes);
          tma_load_3d(dst, &tm_k, &sh.full[s], 0, n_begin + t * kTile, bh);
          if (kSepValues) tma_load_3d(dst + kValueOff, &tm_v, &sh.full[s], 0, n_begin + t * kTile, bh);
          issued = t + 1;
          FLAREPP_TR(tr_on, kTrLoad, t);
        }
      }
      if (kNormKeys) {
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        const int tn = t - kLag;
        if (ok && tn >= 0) {
          ok = normalise_part<D, kStages>(sh, sStage, kStageBytes, tn, 0, lane);
          FLAREPP_TR(tr_on && ok && lane == 0, kTrNorm, tn);
        }
      }
    }
    if (lane == 0 && *(volatile int*)&sh.abort) {
      // let the copies still in flight land before the CTA leaves
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait(&sh.full[t % kStages], (t / kStages) & 1, sh.wait_limit);
      mbar_wait(&sh.q_full, 0, sh.wait_limit);
    }
  } else if (warp < kWarpNorm) {
    // ---------------------------------- MMA of column half hf of slot kk
    {  // the whole warp runs the issuing loop; one elected lane issues
      const int kk = (warp - kWarpIssue) >> 1, hf = (warp - kWarpIssue) & 1;
      const uint32_t aOnes = smem_u32(sOnes);
      const uint32_t idS = idesc_bf16(128, 64, false, false);
      const uint32_t idO = idesc_bf16(128, L::kNo, false, true);
      const uint32_t rows_off = hf * 64 * L::kRowBytes;  // first token row of the half in a tile
      constexpr uint32_t kLo = 0u, kAll = 0xFFFFFFFFu;
      // The plan in scalars (a slot index only known at run time would put the
      // plan in local memory, and every step would wait for an L1 load):
      // slot kk's step j works on tile t0 + dt * j (in the lanes mode lanes
      // 64-127 take the next tile as well).
      const bool lanes = sp.mode == kLanes;
      const int nsteps = kk ? sp.steps[1] : sp.steps[0];
      const int t0 = lanes ? 2 * kk : (sp.mode == kStreams ? kk : 0);
      const int dt = lanes ? 4 : (sp.mode == kStreams ? 2 : 1);
      const uint32_t dS = tmem + kk * kSlotCols + 64 * hf;
      const uint32_t tQ = tmem + kk * kSlotCols + kColQ;
      const uint32_t dO = tmem + kk * kSlotCols + kColO + hf * L::kNo;
      const uint32_t aP = tmem + kk * kSlotCols + 64 * hf;
      auto ready = [&](int t) -> bool {
        return warp_wait(sh, kNormKeys ? &sh.norm[t % kStages] : &sh.full[t % kStages], (t / kStages) & 1);
      };
      // Descriptors of stage 0, built once; stage s is s * kStageBytes further:
      // the key descriptor's start address moves by that much, and so does the
      // value descriptor's, whose distance to the ones tile (its leading byte
      // offset field) shrinks by as much. Both fields stay in range, so one
      // 64-bit add per stage moves them.
      const uint64_t dK0 = L::kmajor(smem_u32(sStage) + rows_off, 0);
      const uint64_t dV0 = L::values1(smem_u32(sStage) + kValueOff, aOnes, 4 * hf);
      constexpr uint64_t kStep = kStageBytes >> 4;
      constexpr uint64_t kVStep = kStep - (kStep << 16);  // modulo 2^64
      auto key_desc = [&](int t) { return dK0 + static_cast<uint64_t>(t % kStages) * kStep; };
      auto val_desc = [&](int t) { return dV0 + static_cast<uint64_t>(t % kStages) * kVStep; };
      // scores of the half's 64 token columns of tile t (and t + 1 in the
      // lanes mode); the latent queries (A) are read from TMEM, the keys (B)
      // from the staged tile
      // tile t (and t + 1 in the lanes mode) staged and normalised; waited
      // for while the issuer has nothing else to do
      auto tile_ready = [&](int t) -> bool {
        if (!ready(t)) return false;
        return !(lanes && t + 1 < T) || ready(t + 1);
      };
      auto issue_s = [&](int t) -> bool {
        if (lanes) {
          const bool has_b = t + 1 < T;
          tc_fence_after();
          const uint64_t ka = key_desc(t);
#pragma unroll
          for (int q = 0; q < D / 16; ++q)
            mma_ts_masked_elect(dS, tQ + q * 8, L::adv(ka, 32 * q), idS, q > 0, kLo, kLo, kAll, kAll);
          if (has_b) {
            const uint64_t kb = key_desc(t + 1);
#pragma unroll
            for (int q = 0; q < D / 16; ++q)
              mma_ts_masked_elect(dS, tQ + q * 8, L::adv(kb, 32 * q), idS, q > 0, kAll, kAll, kLo, kLo);
          }
        } else {
          tc_fence_after();
          const uint64_t ka = key_desc(t);
#pragma unroll
          for (int q = 0; q < D / 16; ++q) mma_ts_elect(dS, tQ + q * 8, L::adv(ka, 32 * q), idS, q > 0);
        }
        mma_commit_elect(&sh.s_full[kk][hf]);
        return true;
      };
      // O_hf (+)= P_hf [V | 1]_hf for tile t (and t + 1): slices 4hf .. 4hf+3
      // of the tile, P of the half at column 64hf of the slot
      auto issue_pv = [&](int t, uint32_t first) {
        const uint64_t va = val_desc(t);
        if (lanes) {
          const bool has_b = t + 1 < T;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mma_ts_masked_elect(dO, aP + i * 8, L::adv(va, i * 2 * L::kAtom), idO, i > 0 ? 1u : first, kLo, kLo, kAll,
                          kAll);
          if (has_b) {
            const uint64_t vb = val_desc(t + 1);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              mma_ts_masked_elect(dO, aP + i * 8, L::adv(vb, i * 2 * L::kAtom), idO, i > 0 ? 1u : first, kAll, kAll, kLo,
                            kLo);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) mma_ts_elect(dO, aP + i * 8, L::adv(va, i * 2 * L::kAtom), idO, i > 0 ? 1u : first);
        }
      };
      // the stage(s) of tile t can be refilled once this thread's products of
      // them are done (every issuing thread that read them releases)
      auto release = [&](int t) {
        mma_commit_elect(&sh.empty[t % kStages]);
        if (lanes && t + 1 < T) mma_commit_elect(&sh.empty[(t + 1) % kStages]);
      };
      bool ok = nsteps > 0 && warp_wait(sh, &sh.q_tmem, 0) && tile_ready(t0);
      tc_fence_after();
      if (ok) ok = issue_s(t0);
      // Per step: the products that read P, then at once the next step's
      // scores (its tile was waited for before P was), then the release of
      // the tile: the path from P to the next scores holds no wait and one
      // commit.
      for (int j = 0, t = t0; ok && j < nsteps; ++j, t += dt) {
        const bool more = j + 1 < nsteps;
        if (more && !tile_ready(t + dt)) break;
        if (!warp_wait(sh, &sh.p_full[kk][hf], j & 1)) break;
        FLAREPP_TR(tr_on && lane == 0, kTrIssue + 2 * kk + hf, 3 * j);
        tc_fence_after();
        issue_pv(t, j > 0 ? 1u : 0u);
        FLAREPP_TR(tr_on && lane == 0, kTrIssue + 2 * kk + hf, 3 * j + 1);
        if (more) ok = issue_s(t + dt);
        release(t);
        FLAREPP_TR(tr_on && lane == 0, kTrIssue + 2 * kk + hf, 3 * j + 2);
      }
      // every MMA of this CTA completes before TMEM is released
      mma_commit_elect(&sh.drain);
      mbar_wait(&sh.drain, 0, sh.wait_limit);
    }
  } else if (warp == kWarpNorm || warp >= kWarpSoftmax + 8) {
    // ------------------------------------------- N0 of the synthesis keys
    if (kNormKeys) {
      const int part = warp == kWarpNorm ? 1 : warp - (kWarpSoftmax + 6);  // 1, 2, 3
      for (int t = 0; t < T; ++t) {
        if (!normalise_part<D, kStages>(sh, sStage, kStageBytes, t, part, lane)) break;
        FLAREPP_TR(tr_on && lane == 0, kTrNorm + part, t);
      }
    }
  } else if (warp >= kWarpSoftmax && warp < kWarpSoftmax + 8) {
    // ------------------------------------------------- softmax + epilogue
    const int tid = threadIdx.x - 32 * kWarpSoftmax;  // 0..255
    const int hf = tid >> 7;                           // column half
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int lanes_half = sp.mode == kLanes ? (row >> 6) : 0;
    const float c = rsqrtf((float)D) * kLog2e;
#ifdef FLAREPP_TRACE
    const bool tr_sm = tr_on && lane == 0 && (warp == kWarpSoftmax || warp == kWarpSoftmax + 4);
#endif
    float r[2] = {-INFINITY, -INFINITY}, ro[2] = {-INFINITY, -INFINITY};  // references of P and of O
    bool acc[2] = {false, false};
    bool ok = true;
    if (hf == 0) {
      // latent query row `row` of each slot's block from the staged tile into
      // the slot's Q columns (lane = latent row, bf16 pairs)
      ok = wait_or_abort(sh, &sh.q_full, 0);
      if (ok) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const unsigned char* src = sQ + (sp.mode == kPair ? k * L::kTileBytes : 0);
          uint32_t w[D / 2];
#pragma unroll
          for (int cc = 0; cc < D / 8; ++cc) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + L::chunk_offset(row, cc));
            w[4 * cc] = v.x; w[4 * cc + 1] = v.y; w[4 * cc + 2] = v.z; w[4 * cc + 3] = v.w;
          }
          const uint32_t tQ = tmem + lane_base + k * kSlotCols + kColQ;
          if (D == 32) tmem_st16(tQ, *reinterpret_cast<uint32_t(*)[16]>(w));
          else tmem_st8(tQ, *reinterpret_cast<uint32_t(*)[8]>(w));
        }
        tmem_wait_st();
      }
      warp_arrive(&sh.q_tmem);
    }
    for (int j = 0; ok && j < jmax; ++j) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (!ok || j >= sp.steps[k]) continue;
        const uint32_t tS = tmem + lane_base + k * kSlotCols + 64 * hf;
        const uint32_t tO = tmem + lane_base + k * kSlotCols + kColO + hf * Layout<D>::kNo;
        if (!wait_or_abort(sh, &sh.s_full[k][hf], j & 1)) { ok = false; continue; }
        FLAREPP_TR(tr_sm, kTrSoftmax + hf, 4 * j + 2 * k);
        tc_fence_after();
        const int t = slot_tile(sp, k, j) + lanes_half;
        bool wrote = false;
        if (t < T) {
          const int valid = min(kTile, n_end - (n_begin + t * kTile)) - 64 * hf;
          if (valid > 0) {
            softmax_half(tS, min(valid, 64), c, r[k]);
            wrote = true;
          } else {
            // no token in this half of the last tile: P = 0
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
            tmem_st32(tS, z);
          }
        }
        finish_half<D>(&sh.p_full[k][hf], tO, r[k], ro[k], acc[k]);
        FLAREPP_TR(tr_sm, kTrSoftmax + hf, 4 * j + 2 * k + 1);
        if (wrote) acc[k] = true;
      }
    }
    // every product is complete before the stage buffers are reused as
    // scratch below
    if (ok) ok = wait_or_abort(sh, &sh.drain, 0);
    tc_fence_after();
    FLAREPP_TR(tr_on && tid == 0, kTrEpi, 0);

    // 1) each softmax stream's (L, Z) into shared memory: stream e =
    //    256 hf + 128 k + row
    constexpr int kZs = D + 1;  // padded row stride
    float* scr_l = reinterpret_cast<float*>(sStage);  // [512]
    float* scr_z = scr_l + 512;                       // [512][D + 1]
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float o[D];
      const float l = load_acc<D>(tmem + lane_base + k * kSlotCols + kColO + hf * Layout<D>::kNo, o);
      const int e = 256 * hf + 128 * k + row;
      const bool any = ok && acc[k] && l > 0.f;  // a stream with no token never wrote its accumulator
      const float inv = any ? 1.f / l : 0.f;
      scr_l[e] = any ? (ro[k] + __log2f(l)) * kLn2 : -INFINITY;
#pragma unroll
      for (int d = 0; d < D; ++d) scr_z[e * kZs + d] = any ? o[d] * inv : 0.f;
    }
    softmax_groups_sync();

    // 2) one partial result per (latent row, split): the CTA's streams of a
    //    row merged first (Appendix B.3 schedule over the streams). Stream e
    //    belongs to latent row (e & 127) of block qt of slot (e >> 7) & 1; in
    //    the lanes mode row r and r + 64 hold the same latent.
    {
      const int nwriters = sp.mode == kLanes ? 64 : (sp.mode == kStreams ? 128 : 256);
      const int nent = 512 / nwriters;
      for (int e = tid; e < nwriters; e += 256) {
        const int r_w = e & 127;
        const int qt_w = sp.mode == kPair && (e >> 7) ? sp.qt[1] : sp.qt[0];
        const int latent_w = qt_w * kTile + r_w;
        if (latent_w >= p.M) continue;
        float lmax = -INFINITY;
        for (int i = 0; i < nent; ++i) lmax = fmaxf(lmax, scr_l[e + i * nwriters]);
        float u[D], dsum = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) u[d] = 0.f;
        for (int i = 0; i < nent; ++i) {
          const float li = scr_l[e + i * nwriters];
          const float w = li == -INFINITY ? 0.f : __expf(li - lmax);
          dsum += w;
#pragma unroll
          for (int d = 0; d < D; ++d) u[d] = fmaf(w, scr_z[(e + i * nwriters) * kZs + d], u[d]);
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
    FLAREPP_TR(tr_on && tid == 0, kTrEpi, 1);
    if (tid == 0) {
      const unsigned prev = atomicAdd(p.counters + grp, 1u);
      sh.last = prev == (unsigned)(p.splits - 1);
    }
    softmax_groups_sync();
    FLAREPP_TR(tr_on && tid == 0, kTrEpi, 2);
    if (sh.last) {
      __threadfence();
      if (tid == 0) p.counters[grp] = 0u;  // ready for the next call
      // 3) the last CTA of the group merges the splits (Appendix B.3:
      //    L_max, d_s = exp(L_s - L_max), U = sum d_s Z_s, Z = U / d), with
      //    `tpr` threads per latent row sharing the splits
      const int rows = sp.mode == kLanes ? 64 : (sp.mode == kStreams ? 128 : 256);
      const int tpr = 256 / rows;
      const int rg = tid / tpr, part = tid % tpr;
      const int qt_f = sp.mode == kPair && (rg >> 7) ? sp.qt[1] : sp.qt[0];
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
        const size_t rr = base + (size_t)sidx * kTile;
        const float ls = __ldcg(p.part_l + rr);
        const float w = ls == -INFINITY ? 0.f : __expf(ls - lmax);
        dsum += w;
        const float4* zr = reinterpret_cast<const float4*>(p.part_z + rr * D);
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
        if (pass_gated(kKind)) {
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
  FLAREPP_TR(tr_on && threadIdx.x == 0, kTrStart, 1);
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ----------------------------------------------------------- decode kernel
struct DecodeParams {
  int N, M, H, BH;
  int tiles_per_cta;   // consecutive token tiles per CTA
  int ctas_per_head;   // > 0: a CTA's tiles lie in one head; 0: tiles in flattened (head, tile) order
  int heads;           // Q/Z slots in shared memory: the most heads one CTA's tiles span
  int q_by_head;       // routing queries [H][M][D] (1) or [BH][M][D] (0)
  __nv_bfloat16* out;  // [BH][N][D]
  int fail_wait;       // test only: P barrier of slot 0, half 0 expects one arrival too many
};

// Token-tile ring depth of the decode kernel: a compile-time constant, so
// that the ring index and phase of a tile cost no division on the issuing
// threads. With Q and Z of M <= 512 routes resident it still fits.
constexpr int kDecodeStages = kMaxStages;
// At most this many heads' Q and Z per CTA, within this much shared memory.
constexpr int kDecodeHeads = 4;
constexpr int kDecodeSmemLimit = 220 * 1024;
template <int D>
__host__ __device__ constexpr int decode_smem_bytes(int M, int heads) {
  return 1024 + (2 * heads * ((M + kTile - 1) / kTile) + kDecodeStages + 1) * (int)Layout<D>::kTileBytes;
}
static_assert(decode_smem_bytes<32>(512, 1) <= kDecodeSmemLimit, "decode ring does not fit next to Q and Z");

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
  const uint32_t head_bytes = chunks * L::kTileBytes;      // Q (or Z) of one head
  constexpr int stages = kDecodeStages;
  unsigned char* sQ = smem;                                // [heads][chunks][128][D]
  unsigned char* sZ = smem + p.heads * head_bytes;         // [heads][chunks][128][D]
  unsigned char* sK = smem + 2 * p.heads * head_bytes;     // [stages][128][D]
  unsigned char* sOnes = sK + stages * L::kTileBytes;      // [128][D]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The CTA's token tiles: T consecutive tiles of the flattened (head, tile)
  // order, from tile `first` of head h0. They span `nheads` heads, whose Q and
  // Z all stay resident; local tile t belongs to head h0 + head_slot(t).
  const int n_tiles = (p.N + kTile - 1) / kTile;
  long long g0;
  int T;
  if (p.ctas_per_head > 0) {
    const int hh = blockIdx.x / p.ctas_per_head, j = blockIdx.x - hh * p.ctas_per_head;
    g0 = (long long)hh * n_tiles + (long long)j * p.tiles_per_cta;
    T = max(0, min(p.tiles_per_cta, n_tiles - j * p.tiles_per_cta));
  } else {
    g0 = (long long)blockIdx.x * p.tiles_per_cta;
    T = (int)max(0LL, min((long long)p.tiles_per_cta, (long long)p.BH * n_tiles - g0));
  }
  const int h0 = (int)(g0 / n_tiles);
  const int first = (int)(g0 - (long long)h0 * n_tiles);
  const int nheads = T > 0 ? (first + T - 1) / n_tiles + 1 : 1;
  if (nheads > p.heads) {
    // more heads than the plan made room for: record it, run nothing
    if (threadIdx.x == 0) atomicOr(&g_tc_error, kErrBadState);
    return;
  }
  int bnd[kDecodeHeads];  // first local tile of head slot i >= 1; past every tile when absent
#pragma unroll
  for (int i = 0; i < kDecodeHeads; ++i) bnd[i] = i > 0 && i < nheads ? i * n_tiles - first : INT_MAX;
  auto head_slot = [&](int t) {
    int hs = 0;
#pragma unroll
    for (int i = 1; i < kDecodeHeads; ++i) hs += t >= bnd[i] ? 1 : 0;
    return hs;
  };
  // Schedule: each column half of a slot owns whole token tiles and runs over
  // all M routes of its tile in `nsub` steps of 64 routes, carrying its online
  // softmax over M from one step to the next, so its accumulator ends as a
  // whole output row and the two halves never exchange data. Step u of slot k
  // works on tile pair g = 2 (u / nsub) + k: half hf takes local tile
  // 2g + hf, routes 64 (u % nsub) .. +63.
  const int nsub = (p.M + 63) / 64;
  int steps[2];
  {
    const int G = (T + 1) / 2;
    for (int k = 0; k < 2; ++k) steps[k] = (G > k ? (G - k + 1) / 2 : 0) * nsub;
  }
  const int umax = max(steps[0], steps[1]);
  // local token tile of half hf of slot k's step u (may be past T when T is odd)
  auto tile_of = [&](int k, int u, int hf) { return 2 * (2 * (u / nsub) + k) + hf; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);  // a tile is read by one issuing thread
    }
    mbar_init(&sh.q_full, 1);
    for (int k = 0; k < 2; ++k)
      for (int hf = 0; hf < 2; ++hf) {
        mbar_init(&sh.s_full[k][hf], 1);
        mbar_init(&sh.p_full[k][hf], 4 + (p.fail_wait && k == 0 && hf == 0 ? 1 : 0));
        mbar_init(&sh.o_full[k][hf], 1);
      }
    mbar_init(&sh.drain, 4);
    sh.wait_limit = p.fail_wait ? kTestWaitLimit : kWaitLimit;
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= kWarpSoftmax && warp < kWarpSoftmax + 8) fill_ones<D>(sOnes, threadIdx.x - 32 * kWarpSoftmax, 256);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
#ifdef FLAREPP_TRACE
  const bool tr_on = blockIdx.x == 0 && g_trace_pass == 3;
#endif
  FLAREPP_TR(tr_on && threadIdx.x == 0, kTrStart, 0);

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_z);
      mbar_arrive_expect_tx(&sh.q_full, 2 * nheads * head_bytes);
      for (int hs = 0; hs < nheads; ++hs) {
        const int bh = h0 + hs;
        for (int ch = 0; ch < chunks; ++ch) {
          const uint32_t off = hs * head_bytes + ch * L::kTileBytes;
          tma_load_3d(sQ + off, &tm_q, &sh.q_full, 0, ch * kTile, p.q_by_head ? bh % p.H : bh);
          tma_load_3d(sZ + off, &tm_z, &sh.q_full, 0, ch * kTile, bh);
        }
      }
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % stages;
        if (t >= stages && !wait_or_abort<true>(sh, &sh.empty[s], ((t / stages) - 1) & 1)) break;
        const int hs = head_slot(t);
        mbar_arrive_expect_tx(&sh.full[s], L::kTileBytes);
        tma_load_3d(sK + s * L::kTileBytes, &tm_k, &sh.full[s], 0, (first + t - hs * n_tiles) * kTile, h0 + hs);
        issued = t + 1;
        FLAREPP_TR(tr_on, kTrLoad, t);
      }
      if (*(volatile int*)&sh.abort) {
        for (int t = max(0, issued - stages); t < issued; ++t)
          mbar_wait(&sh.full[t % stages], (t / stages) & 1, sh.wait_limit);
        mbar_wait(&sh.q_full, 0, sh.wait_limit);
      }
    }
  } else if (warp < kWarpNorm) {
    {  // the whole warp runs the issuing loop; one elected lane issues
      const int kk = (warp - kWarpIssue) >> 1, hf = (warp - kWarpIssue) & 1;
      const uint32_t aZ = smem_u32(sZ), aOnes = smem_u32(sOnes);
      const uint32_t idO = idesc_bf16(128, L::kNo, false, true);
      // descriptors built once; an MMA moves them with one add (a thread
      // spends its issue slots on every instruction between MMAs). Routes
      // 64b .. 64b+63 start 64b rows into the chunked Q (and Z) tiles.
      const uint64_t dK0 = L::kmajor(smem_u32(sK), 0);
      const uint64_t dQ0 = L::kmajor(smem_u32(sQ), 0);
      const uint32_t idS64 = idesc_bf16(128, 64, false, false);
      const uint32_t dS = tmem + kk * kSlotCols + 64 * hf;
      const uint32_t dO = tmem + kk * kSlotCols + kColO + hf * L::kNo;
      // scores of local tile t against routes 64b .. 64b+63 of its head, whose
      // Q and Z sit `hoff` bytes into their arrays
      // the K tile of local tile t staged (waited for at its first route
      // block, while the issuer has nothing else to do)
      auto tile_wait = [&](int t, int b) -> bool {
        if (t >= T || b != 0) return true;
        return warp_wait(sh, &sh.full[t % stages], (t / stages) & 1);
      };
      auto issue_s = [&](int t, int b, uint32_t hoff) -> bool {
        if (t < T) {
          const int s = t % stages;
          tc_fence_after();
          const int width = min(64, p.M - 64 * b);
          const uint64_t a = L::adv(dK0, s * L::kTileBytes), bq = L::adv(dQ0, hoff + b * 64 * L::kRowBytes);
          const uint32_t id = width >= 64 ? idS64 : idesc_bf16(128, width, false, false);
#pragma unroll
          for (int q = 0; q < D / 16; ++q) mma_ss_elect(dS, L::adv(a, 32 * q), L::adv(bq, 32 * q), id, q > 0);
        }
        mma_commit_elect(&sh.s_full[kk][hf]);
        // the tile's last read: its stage may be refilled
        if (t < T && b == nsub - 1) mma_commit_elect(&sh.empty[t % stages]);
        return true;
      };
      // O_hf (+)= P_hf [Z | 1] over the route slices of block b
      auto issue_pv = [&](int t, int b, uint32_t hoff) {
        if (t >= T) return;
        const int nsl = min(64, p.M - 64 * b) / 16;
        const uint64_t v = L::values1(aZ + hoff + (b >> 1) * L::kTileBytes, aOnes, 4 * (b & 1));
        const uint32_t aP = tmem + kk * kSlotCols + 64 * hf;
        const uint32_t first = b > 0 ? 1u : 0u;
        if (nsl == 4) {
#pragma unroll
          for (int i = 0; i < 4; ++i) mma_ts_elect(dO, aP + i * 8, L::adv(v, i * 2 * L::kAtom), idO, i > 0 ? 1u : first);
        } else {
          for (int i = 0; i < nsl; ++i) mma_ts_elect(dO, aP + i * 8, L::adv(v, i * 2 * L::kAtom), idO, i > 0 ? 1u : first);
        }
      };
      // the step's tile and route block, advanced without a division
      int t = tile_of(kk, 0, hf), b = 0;
      uint32_t hoff = head_slot(t) * head_bytes;
      const int nsteps = kk ? steps[1] : steps[0];  // no run-time array index: steps stays in registers
      bool ok = nsteps > 0 && warp_wait(sh, &sh.q_full, 0) && tile_wait(t, b);
      if (ok) ok = issue_s(t, b, hoff);
      // Per step: the products that read P, then at once the next step's
      // scores (whose tile was waited for before P was).
      for (int u = 0; ok && u < nsteps; ++u) {
        int tn = t, bn = b + 1;
        uint32_t hn = hoff;
        if (bn == nsub) {
          bn = 0;
          tn = t + 4;
          hn = head_slot(tn) * head_bytes;
        }
        const bool more = u + 1 < nsteps;
        if (more && !tile_wait(tn, bn)) break;
        if (!warp_wait(sh, &sh.p_full[kk][hf], u & 1)) break;
        FLAREPP_TR(tr_on && lane == 0, kTrIssue + 2 * kk + hf, 3 * u);
        tc_fence_after();
        issue_pv(t, b, hoff);
        FLAREPP_TR(tr_on && lane == 0, kTrIssue + 2 * kk + hf, 3 * u + 1);
        if (more) ok = issue_s(tn, bn, hn);
        else mma_commit_elect(&sh.o_full[kk][hf]);
        FLAREPP_TR(tr_on && lane == 0, kTrIssue + 2 * kk + hf, 3 * u + 2);
        t = tn;
        b = bn;
        hoff = hn;
      }
      mma_commit_elect(&sh.drain);
      mbar_wait(&sh.drain, 0, sh.wait_limit);
    }
  } else if (warp >= kWarpSoftmax && warp < kWarpSoftmax + 8) {
    const int tid = threadIdx.x - 32 * kWarpSoftmax;  // 0..255
    const int hf = tid >> 7;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float c = rsqrtf((float)D) * kLog2e;
#ifdef FLAREPP_TRACE
    const bool tr_sm = tr_on && lane == 0 && (warp == kWarpSoftmax || warp == kWarpSoftmax + 4);
#endif
    float r[2] = {-INFINITY, -INFINITY}, ro[2] = {-INFINITY, -INFINITY};
    bool acc[2] = {false, false};
    // out = O / rowsum of this half's accumulator, for its own token tile t
    auto emit = [&](int k, int t, bool live) {
      if (!live || t >= T) return;
      float z[D];
      const float l = load_acc<D>(tmem + lane_base + k * kSlotCols + kColO + hf * Layout<D>::kNo, z);
      const int hs = head_slot(t);
      const int tok = (first + t - hs * n_tiles) * kTile + row;
      if (tok < p.N) {
        const float inv = 1.f / l;
#pragma unroll
        for (int d = 0; d < D; ++d) z[d] *= inv;
        store_row<D>(p.out + ((size_t)(h0 + hs) * p.N + tok) * D, z);
      }
    };
    bool ok = true;
    // the step's route block (the same for both slots) and each slot's tile
    int b = 0;
    int tk[2] = {tile_of(0, 0, hf), tile_of(1, 0, hf)};
    for (int u = 0; u < umax; ++u) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (u >= steps[k]) continue;
        const uint32_t tS = tmem + lane_base + k * kSlotCols + 64 * hf;
        const uint32_t tO = tmem + lane_base + k * kSlotCols + kColO + hf * Layout<D>::kNo;
        ok = ok && wait_or_abort(sh, &sh.s_full[k][hf], u & 1);
        FLAREPP_TR(tr_sm, kTrSoftmax + hf, 4 * u + 2 * k);
        tc_fence_after();
        if (b == 0) {
          // the previous tile's products are in: its output goes out before
          // this step's products overwrite the accumulator
          if (u > 0) emit(k, tk[k] - 4, ok);
          r[k] = -INFINITY;
          acc[k] = false;
        }
        if (!ok) continue;
        const int valid = tk[k] < T ? min(64, p.M - 64 * b) : 0;
        if (valid > 0) softmax_half(tS, valid, c, r[k]);
        finish_half<D>(&sh.p_full[k][hf], tO, r[k], ro[k], acc[k]);
        FLAREPP_TR(tr_sm, kTrSoftmax + hf, 4 * u + 2 * k + 1);
        if (valid > 0) acc[k] = true;
      }
      if (++b == nsub) {
        b = 0;
        tk[0] += 4;
        tk[1] += 4;
      }
    }
    // the last tile of each slot
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (steps[k] == 0) continue;
      const bool done = ok && wait_or_abort(sh, &sh.o_full[k][hf], 0);
      tc_fence_after();
      emit(k, tile_of(k, steps[k] - 1, hf), done);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  FLAREPP_TR(tr_on && threadIdx.x == 0, kTrStart, 1);
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host
template <int D, int kKind>
size_t split_smem() {
  const size_t stage = (pass_separate_values(kKind) ? 2 : 1) * (size_t)Layout<D>::kTileBytes;
  return 1024 + 3 * (size_t)Layout<D>::kTileBytes + split_stages<D, kKind>() * stage;
}

template <int D>
size_t decode_smem(int M, int heads) {
  return (size_t)decode_smem_bytes<D>(M, heads);
}

template <int D, int kKind>
cudaError_t launch_split(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const SplitParams& a,
                         dim3 grid, cudaStream_t stream, const char* what, const char** failed) {
  const size_t smem = split_smem<D, kKind>();
  *failed = "cudaFuncSetAttribute(split_kernel)";
  cudaError_t e = cudaFuncSetAttribute(split_kernel<D, kKind>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  split_kernel<D, kKind><<<grid, kThreads, smem, stream>>>(mq, mk, mv, a);
  *failed = what;
  return cudaGetLastError();
}

// The passes of one call. The synthesis pass depends on the variant: shared
// keys and values (eq. 19), separate values (eq. 11), the ungated synthesis of
// the simplified variant (eq. 20, an encode-kind pass with per-head queries
// writing Q), or none (FLARE, eq. 3, whose queries are the caller's). Encode
// and decode are the same for all four.
template <int D>
cudaError_t forward_d(const DeviceProblem& pr, const TcPlan& pl, const TcWorkspace& ws, cudaEvent_t* ev,
                      cudaStream_t stream, const char** failed) {
  const int BH = pr.B * pr.H;
  const bool flare = pr.variant == kVariantFlare;
  cudaError_t e;
  CUtensorMap m_seed, m_ks, m_vs, m_qenc, m_k, m_v, m_qdec, m_zdec;
  const int qbox = pr.M <= 64 ? 64 : kTile;
  // routing queries: the caller's per-head set (FLARE) or the synthesis output
  const void* qsrc = flare ? pr.Q : ws.q;
  const int qplanes = flare ? pr.H : BH;
  *failed = "cuTensorMapEncodeTiled";
  if (!make_map(&m_qenc, qsrc, D, pr.M, qplanes, qbox) || !make_map(&m_k, pr.K, D, pr.N, BH, kTile) ||
      !make_map(&m_v, pr.V, D, pr.N, BH, kTile) || !make_map(&m_qdec, qsrc, D, pr.M, qplanes, kTile) ||
      !make_map(&m_zdec, ws.z, D, pr.M, BH, kTile))
    return cudaErrorInvalidValue;
  if (!flare) {
    const void* vs = pr.variant == kVariantFlarePP ? pr.Ks : pr.Vs;
    if (!make_map(&m_seed, pr.Qseed, D, pr.M, pr.H, qbox) || !make_map(&m_ks, pr.Ks, D, pr.N, BH, kTile) ||
        !make_map(&m_vs, vs, D, pr.N, BH, kTile))
      return cudaErrorInvalidValue;
  }

  const dim3 grid(pl.splits, pl.qgroups, BH);
  SplitParams sp{};
  sp.N = pr.N; sp.M = pr.M; sp.H = pr.H;
  sp.fail_wait = 0;
  sp.qtiles = pl.tiles; sp.splits = pl.splits; sp.split_len = pl.split_len;
  sp.part_z = ws.part_z; sp.part_l = ws.part_l;

  if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) { *failed = "cudaEventRecord"; return e; }
  // synthesis (a1-a3)
  if (!flare) {
    SplitParams a = sp;
    a.counters = ws.counters;
    a.q_by_head = 1;
    a.out = static_cast<__nv_bfloat16*>(ws.q);
    a.fail_wait = pr.fail_wait == 1;
    if (pr.variant == kVariantSimplified) {
      a.dbg_a = pr.dbg_q;  // Q = Qd, as rounded
      e = launch_split<D, kPassEncode>(m_seed, m_ks, m_vs, a, grid, stream, "launch synthesis", failed);
    } else {
      a.qf = static_cast<const __nv_bfloat16*>(pr.Qf);
      a.gate = pr.gate;
      a.dbg_a = pr.dbg_qd;
      a.dbg_b = pr.dbg_q;
      e = pr.variant == kVariantUnshared
              ? launch_split<D, kPassSynthSeparate>(m_seed, m_ks, m_vs, a, grid, stream, "launch synthesis", failed)
              : launch_split<D, kPassSynthShared>(m_seed, m_ks, m_ks, a, grid, stream, "launch synthesis", failed);
    }
    if (e != cudaSuccess) return e;
  }
  if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) { *failed = "cudaEventRecord"; return e; }
  // encode (a4-a5)
  {
    SplitParams a = sp;
    a.counters = ws.counters + (size_t)BH * pl.qgroups;
    a.q_by_head = flare ? 1 : 0;
    a.fail_wait = pr.fail_wait == 2;
    a.out = static_cast<__nv_bfloat16*>(ws.z);
    a.dbg_a = pr.dbg_z;
    a.dbg_b = pr.dbg_l;
    if ((e = launch_split<D, kPassEncode>(m_qenc, m_k, m_v, a, grid, stream, "launch encode", failed)) != cudaSuccess)
      return e;
  }
  if (ev && (e = cudaEventRecord(ev[2], stream)) != cudaSuccess) { *failed = "cudaEventRecord"; return e; }
  // decode (a6)
  {
    DecodeParams d{};
    d.N = pr.N; d.M = pr.M; d.H = pr.H; d.BH = BH;
    d.tiles_per_cta = pl.decode_tiles_per_cta;
    d.ctas_per_head = pl.decode_ctas_per_head;
    d.heads = pl.decode_heads;
    d.q_by_head = flare ? 1 : 0;
    d.out = static_cast<__nv_bfloat16*>(pr.out);
    d.fail_wait = pr.fail_wait == 3;
    const size_t smem = decode_smem<D>(pr.M, pl.decode_heads);
    *failed = "cudaFuncSetAttribute(decode)";
    if ((e = cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    decode_kernel<D><<<pl.decode_ctas, kThreads, smem, stream>>>(m_k, m_qdec, m_zdec, d);
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
  // decode: one CTA per SM over consecutive token tiles. In the flattened
  // (head, tile) order every SM gets the same number of tiles, if each CTA
  // has room for the Q and Z of every head its tiles span; otherwise a CTA's
  // tiles stay within one head, split by the same cost model as the encode.
  const long long total = BH * n_tiles;
  const int per_flat = (int)std::max(2LL, (total + std::max(1, sms) - 1) / std::max(1, sms));
  const int heads_flat = (per_flat - 1 + n_tiles - 1) / n_tiles + 1;
  const int smem_flat = D == 16 ? tc::decode_smem_bytes<16>(M, heads_flat) : tc::decode_smem_bytes<32>(M, heads_flat);
  if (heads_flat <= tc::kDecodeHeads && smem_flat <= tc::kDecodeSmemLimit) {
    pl.decode_tiles_per_cta = per_flat;
    pl.decode_ctas_per_head = 0;
    pl.decode_heads = heads_flat;
    pl.decode_ctas = (int)((total + per_flat - 1) / per_flat);
  } else {
    const int dsplit = tc::choose_splits(BH, n_tiles, std::max(1, sms), 2, 4, 0);
    const int per = (n_tiles + dsplit - 1) / dsplit;
    pl.decode_tiles_per_cta = per;
    pl.decode_ctas_per_head = (n_tiles + per - 1) / per;
    pl.decode_heads = 1;
    pl.decode_ctas = (int)(BH * pl.decode_ctas_per_head);
  }
  return pl;
}

cudaError_t tc_forward(const DeviceProblem& p, const TcPlan& pl, const TcWorkspace& ws, cudaEvent_t* events,
                       cudaStream_t stream, const char** failed_call) {
  return p.D == 16 ? tc::forward_d<16>(p, pl, ws, events, stream, failed_call)
                   : tc::forward_d<32>(p, pl, ws, events, stream, failed_call);
}

// Pipeline trace (trace builds): pass > 0 arms block 0 of that pass and
// clears the stamps, pass == 0 disarms; `host`, when given, receives up to
// n stamps ([role][index] order). Without FLAREPP_TRACE: unsupported.
cudaError_t tc_trace(int pass, unsigned long long* host, int n) {
#ifdef FLAREPP_TRACE
  cudaError_t e = cudaMemcpyToSymbol(tc::g_trace_pass, &pass, sizeof(int));
  if (e != cudaSuccess) return e;
  if (pass > 0) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, tc::g_trace)) != cudaSuccess) return e;
    if ((e = cudaMemset(p, 0, sizeof(tc::g_trace))) != cudaSuccess) return e;
  }
  if (host != nullptr && n > 0) {
    const size_t bytes = std::min(sizeof(tc::g_trace), (size_t)n * sizeof(unsigned long long));
    if ((e = cudaMemcpyFromSymbol(host, tc::g_trace, bytes)) != cudaSuccess) return e;
  }
  return cudaSuccess;
#else
  (void)pass; (void)host; (void)n;
  return cudaErrorNotSupported;
#endif
}

cudaError_t tc_take_error_word(unsigned* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, tc::g_tc_error, sizeof(unsigned));
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(tc::g_tc_error, &zero, sizeof(unsigned));
}

}  // namespace flarepp
