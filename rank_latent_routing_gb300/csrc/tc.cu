// Tensor-core (tcgen05 + TMEM + TMA) kernels of the FLARE++ mixer forward,
// bf16 inputs, fp32 softmax and accumulation.
//
// Two kernels carry the three attention calls of the mixer (FLARE++ paper,
// Section 3.2 eq. 6 and eq. 8):
//
//  * split_kernel — a block of up to 128 latent queries attends over one
//    token range (split) of a head. Scores S = Q K^T land in TMEM; threads
//    run an online softmax over the tokens; P goes back to TMEM in bf16 over
//    the second half of the scores and the tensor core accumulates O += P [V | 1] in TMEM, the
//    appended ones column giving the softmax row sum. Each split's (Z_s, L_s)
//    goes to global memory and the last CTA of a head to arrive merges all
//    splits with the stable log-sum-exp schedule of Appendix B.3 (eq. 29-33);
//    a head with one split writes its result directly. The synthesis instance
//    normalises each staged Ks_raw tile in place (N0, eq. 5), uses it as both
//    keys and values (eq. 19) and ends with the gate (eq. 7):
//    Q = N0(Qf) + g * Qd in fp32, cast to bf16. The encode instance ends with
//    Z (bf16) and L.
//  * decode_kernel — tokens attend over the M routes: Q and Z of the head stay
//    in shared memory for all of the CTA's token tiles; a token tile's scores
//    S = K Q^T are taken 64 routes at a time with an online softmax over M per
//    token, and O += P [Z | 1]; out = O / rowsum in bf16.
//
// One CTA per SM, 512 threads: warp 0 issues TMA loads, warps 1 and 2 issue
// the MMAs of softmax warpgroups 0 and 1 (a whole warp runs each issuing
// loop, one elected lane issues), warps 4, 5, 14 and 15 (one per SM
// sub-partition) normalise a quarter of every synthesis tile each, and two
// softmax warpgroups (warps 6-9 and 10-13) each carry one online-softmax
// stream: in the split kernel warpgroup g takes token rows 64g .. 64g+63 of
// every tile, in the decode kernel every other token tile. Warp w reads TMEM
// lanes 32*(w%4) .. +31, so each sub-partition runs one warp of each stream.
//
// A warpgroup owns 256 TMEM columns: three score buffers of 64 columns, its
// accumulator (D values, the row sum, padding) and, in the split kernel, the
// latent queries (bf16 pairs, the A operand of the score MMAs). Sub-step j of
// a stream uses buffer j % 3: its issuing thread adds the products of step j
// (which read P from buffer j % 3) and at once issues the scores of step j + 3
// into the same buffer, so the softmax finds the scores of its next two steps
// already computed and never waits for the issue-and-complete round trip of
// the tensor core. The tensor core runs one thread's MMAs in order, so the
// new scores overwrite P only after the products have read it.
//
// The softmax is one pass: p = 2^(s*c - r) against a reference r (an integer
// in exp2 units) fixed before the step; the first step of a stream sets r
// from its own max. Whether some p reached 2 is read off the packed bf16
// results (exponent field >= 128 <=> p >= 2, which also catches inf); only
// then does the warp read its scores again, move r to 16 units above the
// ceiling of their max and redo them, and the accumulator is rescaled
// exactly by 2^(r_old - r_new) before the step's products are added, once
// the products of the previous step are complete (the scores of step j + 2
// were issued after them, so their barrier proves it; the issuing thread
// issues two score sets past the end of its stream for this purpose).
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
#include <type_traits>

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
// issuing thread of each stream per step (3 stamps); first softmax warp of
// each stream per step (2 stamps); epilogue phases
enum : int { kTrStart = 0, kTrLoad = 1, kTrNorm = 2, kTrIssue = 6, kTrSoftmax = 10, kTrEpi = 12 };
__device__ __forceinline__ void trace_stamp(bool on, int role, int i) {
  if (on && i >= 0 && i < kTraceLen) g_trace[role][i] = clock64();
}
#define FLAREPP_TR(on, role, i) trace_stamp((on), (role), (i))
#else
#define FLAREPP_TR(on, role, i) ((void)0)
#endif

constexpr int kThreads = 512;
constexpr int kWarpIssue = 1;        // MMA-issuing warps: 1 + stream
constexpr int kWarpNorm = 5;         // N0 of the synthesis tiles: warps 4, 5, 14 and 15
constexpr int kWarpSoftmax = 6;      // first softmax warp (6-13): stream (w - 6) / 4
constexpr int kTile = 128;           // tokens per staged tile; latents per row block
constexpr int kMaxStages = 16;       // token-tile ring depth (upper bound)
constexpr int kBufs = 3;             // score buffers per stream
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kGroupCols = 256;  // stream g owns columns 256g .. 256g+255
constexpr uint32_t kColO = 192;       // the stream's accumulator
constexpr uint32_t kColQ = 240;       // split kernel: the latent queries (bf16 pairs)
constexpr long long kWaitLimit = 2000000000LL;  // clock cycles (~1 s)
// under the test hook that makes one barrier never complete, waits give up
// after ~1 ms, so that the forced timeout ends the call quickly
constexpr long long kTestWaitLimit = 2000000LL;

struct Shared {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t norm[kMaxStages];
  uint64_t q_full;
  uint64_t s_full[2][kBufs];  // scores of stream g in buffer b ready (and the stream's earlier products done)
  uint64_t p_full[2][kBufs];  // P of stream g in buffer b written
  uint64_t o_full[2];         // split: every product of stream g done; decode: a tile's products done
  uint64_t q_tmem[2];         // split: the latent queries are in stream g's columns
  uint64_t drain;             // every MMA of the CTA has completed
  long long wait_limit;       // clock cycles a wait may take before it gives up
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
static_assert(kColO + Layout<32>::kNo <= kColQ && kColQ + 16 <= kGroupCols, "a stream's TMEM columns overlap");
static_assert(kBufs * 64 <= kColO, "score buffers overlap the accumulator");

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
// Exponent field >= 128 in either bf16 half: some p >= 2 (or inf / NaN).
constexpr uint32_t kGrowBits = 0x40004000u;
// When the reference moves it is set this many exp2 units above the tile max,
// so that p <= 2^-16 and the next move waits for the max to grow by 17 units
// (p that small loses nothing: fp32 and bf16 keep their relative precision
// down to 2^-126).
constexpr float kHeadroom = 16.0f;

// P (32 packed words) goes over the second half of a step's 64 score
// columns, so that the first half stays in TMEM for a step that is redone.
constexpr uint32_t kColP = 32;

// p = 2^(s*c - r) of the 64 scores, packed in bf16 pairs over s[0..31]
// (word i is written after scores 2i and 2i + 1 are read, so the scores
// 32..63 stay in s[32..63]); returns the OR of the packed words.
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

__device__ __forceinline__ float max64(const uint32_t (&s)[64]) {
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int i = 0; i < 64; i += 4) {
    m0 = max3(m0, __uint_as_float(s[i]), __uint_as_float(s[i + 1]));
    m1 = max3(m1, __uint_as_float(s[i + 2]), __uint_as_float(s[i + 3]));
  }
  return fmaxf(m0, m1);
}

// Scores of the columns at or past `valid` set to -inf.
__device__ __forceinline__ void mask64(uint32_t (&s)[64], int valid) {
#pragma unroll
  for (int i = 0; i < 64; ++i)
    if (i >= valid) s[i] = __float_as_uint(-INFINITY);
}

// One softmax step of this lane over the 64 score columns at tS, P stored
// over columns 32-63. `kMasked`: columns at or past `valid` count as absent
// (only a stream's last step); `first` (the same in every lane of the warp):
// the stream's first step, whose reference comes from its own max. Later
// steps are done against r in one pass; only if some p reached 2 do those
// lanes move r to 16 units above the ceiling of their max and redo P, with
// the first half of the scores read again from TMEM (the second half is
// still in registers). Returns whether that happened (the same in every
// lane); `r_old` then holds the reference before the move.
template <bool kMasked>
__device__ __forceinline__ bool softmax_step(uint32_t tS, int valid, bool first, float c, float& r, float& r_old) {
  uint32_t s[64];
  tmem_ld64(tS, s);
  tmem_wait_ld_regs(s);
  if (kMasked) mask64(s, valid);
  if (first) r = ceilf(max64(s) * c) + kHeadroom;
  const uint32_t bits = exp_pack(s, c, r);
  tmem_st32(tS + kColP, *reinterpret_cast<uint32_t(*)[32]>(s));
  if (!__any_sync(0xFFFFFFFFu, (bits & kGrowBits) != 0u)) return false;
  tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(s));
  tmem_wait_ld_regs(s);
  if (kMasked) mask64(s, valid);
  r_old = r;
  if ((bits & kGrowBits) != 0u) r = ceilf(max64(s) * c) + kHeadroom;
  tmem_wait_st();  // the first store has landed before it is overwritten
  exp_pack(s, c, r);
  tmem_st32(tS + kColP, *reinterpret_cast<uint32_t(*)[32]>(s));
  return true;
}

// Writes P = 0 (a step with no token).
__device__ __forceinline__ void zero_p(uint32_t tS) {
  uint32_t z[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) z[i] = 0u;
  tmem_st32(tS + kColP, z);
}

// End of a softmax step: if the step was redone (`moved`, the same in every
// lane), the accumulator of each lane whose reference moved from r_old to r
// is brought to the new one, once the stream's previous products are
// complete (`proof`, the barrier of scores issued after them, phase
// `proof_parity`); then P goes to the tensor core (one arrival per warp).
template <int D>
__device__ __forceinline__ bool finish_step(Shared& sh, uint64_t* p_full, uint32_t tO, float r, float r_old,
                                            bool acc, bool moved, uint64_t* proof, uint32_t proof_parity) {
  bool ok = true;
  if (moved) {
    ok = warp_wait(sh, proof, proof_parity);
    tc_fence_after();
    if (ok) rescale_acc<D>(tO, acc && r_old != r ? pow2_neg(r_old - r) : 1.f);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  mbar_arrive_if(p_full, (threadIdx.x & 31) == 0);
  return ok;
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
  unsigned* counters;       // [BH][qtiles]
  int q_by_head;            // latent queries [H][M][D] (1) or [BH][M][D] (0)
  const __nv_bfloat16* qf;  // gated passes: [H][M][D]
  const float* gate;        // gated passes: [H]
  __nv_bfloat16* out;       // gated: Q; encode: Z ([BH][M][D])
  float* dbg_a;             // gated: Qd; encode: Z (as rounded)
  float* dbg_b;             // gated: Q (as rounded); encode: L
  int fail_wait;            // test only: P barrier of stream 0, buffer 0 expects one arrival too many
};

// Epilogue scratch of the split kernel: (L, Z) of 256 softmax streams.
template <int D>
__host__ __device__ constexpr int split_scratch_bytes() {
  return 256 * 4 + 256 * (D + 1) * 4;
}

// Token-tile ring depth of the split kernel: as deep as fits next to the
// latent tile and the ones tile within 180 KB, at most 16 stages. A stage
// holds a key tile, and a value tile unless the keys serve as values. With
// D = 32 and separate values (16 KB stages) that is 10 stages: on a 1M-token
// encode 8, 9 and 11 stages each timed about 1% slower (a 4096-token one
// preferred 8 stages, by a similar margin).
template <int D, int kKind>
__host__ __device__ constexpr int split_stages() {
  constexpr int stage = (pass_separate_values(kKind) ? 2 : 1) * Layout<D>::kTileBytes;
  constexpr int n = (180 * 1024 - 2 * Layout<D>::kTileBytes) / stage;
  return n > kMaxStages ? kMaxStages : n;
}

// The finished row of a latent block (merged over all token splits): the
// gated passes write Q = N0(Qf) + g * u (eq. 7) in bf16, the encode Z = u in
// bf16 and its log-normaliser; the fp32 copies are for stage-level checks.
template <int D, int kKind>
__device__ __forceinline__ void write_final(const SplitParams& p, int bh, int h, int latent, float (&u)[D],
                                            float lse) {
  const size_t orow = (size_t)bh * p.M + latent;
  if (pass_gated(kKind)) {
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
    if (p.dbg_b) p.dbg_b[orow] = lse;
  }
}

template <int D, int kKind, bool kLanes>
__global__ void __launch_bounds__(kThreads, 1)
    split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const SplitParams p) {
  using L = Layout<D>;
  constexpr bool kNormKeys = pass_normalises_keys(kKind);
  constexpr bool kSepValues = pass_separate_values(kKind);
  constexpr int kStages = split_stages<D, kKind>();
  constexpr uint32_t kStageBytes = kSepValues ? 2 * L::kTileBytes : L::kTileBytes;
  constexpr uint32_t kValueOff = kSepValues ? L::kTileBytes : 0;  // value tile within a stage
  // tiles per step: M <= 64 ("lanes" layout): TMEM lanes 64-127 repeat the
  // latents of lanes 0-63 and score the next token tile
  constexpr int kTps = kLanes ? 2 : 1;
  static_assert(kStages * (int)kStageBytes >= split_scratch_bytes<D>(), "epilogue scratch exceeds the stage ring");
  static_assert(kStages > (kBufs + 1) * kTps, "the ring must hold the tiles of the scores issued ahead");
  extern __shared__ unsigned char smem_raw[];
  __shared__ Shared sh;
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  unsigned char* sQ = smem;                                   // [128][D]
  unsigned char* sStage = smem + L::kTileBytes;               // [kStages] x (K, V)
  unsigned char* sOnes = sStage + kStages * kStageBytes;      // [128][D] rows [1, 0, ...]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x, qt = blockIdx.y, bh = blockIdx.z;
  const int h = bh % p.H;
  const int n_begin = split * p.split_len;
  const int n_end = min(p.N, n_begin + p.split_len);
  const int T = n_begin < n_end ? (n_end - n_begin + kTile - 1) / kTile : 0;
  const int U = (T + kTps - 1) / kTps;  // steps of each stream

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 2);  // one release per stream
      mbar_init(&sh.norm[s], 4);   // one arrival per normaliser warp
    }
    mbar_init(&sh.q_full, 1);
    for (int g = 0; g < 2; ++g) {
      for (int b = 0; b < kBufs; ++b) {
        mbar_init(&sh.s_full[g][b], 1);
        // one arrival per softmax warp of the stream (one more under the test hook)
        mbar_init(&sh.p_full[g][b], 4 + (p.fail_wait && g == 0 && b == 0 ? 1 : 0));
      }
      mbar_init(&sh.o_full[g], 1);
      mbar_init(&sh.q_tmem[g], 4);
    }
    mbar_init(&sh.drain, 2);
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
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      if (kSepValues) prefetch_tmap(&tm_v);
      const int qz = p.q_by_head ? h : bh;
      mbar_arrive_expect_tx(&sh.q_full, L::kTileBytes);
      if (kLanes) {
        // the 64 (or fewer) latents twice: lanes 64-127 repeat lanes 0-63
        tma_load_3d(sQ, &tm_q, &sh.q_full, 0, 0, qz);
        tma_load_3d(sQ + L::kTileBytes / 2, &tm_q, &sh.q_full, 0, 0, qz);
      } else {
        tma_load_3d(sQ, &tm_q, &sh.q_full, 0, qt * kTile, qz);
      }
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % kStages;
        if (t >= kStages && !wait_or_abort<true>(sh, &sh.empty[s], ((t / kStages) - 1) & 1)) break;
        unsigned char* dst = sStage + s * kStageBytes;
        mbar_arrive_expect_tx(&sh.full[s], kStageBytes);
        tma_load_3d(dst, &tm_k, &sh.full[s], 0, n_begin + t * kTile, bh);
        if (kSepValues) tma_load_3d(dst + kValueOff, &tm_v, &sh.full[s], 0, n_begin + t * kTile, bh);
        issued = t + 1;
        FLAREPP_TR(tr_on, kTrLoad, t);
      }
      if (*(volatile int*)&sh.abort) {
        // let the copies still in flight land before the CTA leaves
        for (int t = max(0, issued - kStages); t < issued; ++t)
          mbar_wait(&sh.full[t % kStages], (t / kStages) & 1, sh.wait_limit);
        mbar_wait(&sh.q_full, 0, sh.wait_limit);
      }
    }
  } else if (warp == kWarpIssue || warp == kWarpIssue + 1) {
    // ------------------------------------------------ MMAs of stream g
    // The whole warp runs the issuing loop; one elected lane issues. The loop
    // is unrolled over the three score buffers (their TMEM columns and
    // barriers become constants); ring stages and descriptors advance by
    // adds; the wait for the tiles of the scores issued ahead comes before
    // the wait for P, so that from P to the new scores nothing waits.
    const int g = warp - kWarpIssue;
    const uint32_t gbase = tmem + g * kGroupCols;
    const uint32_t tQ = gbase + kColQ, dO = gbase + kColO;
    const uint32_t aOnes = smem_u32(sOnes);
    const uint32_t idS = idesc_bf16(128, 64, false, false);
    const uint32_t idO = idesc_bf16(128, L::kNo, false, true);
    constexpr uint32_t kLo = 0u, kAll = 0xFFFFFFFFu;
    uint64_t* const ready_bar = kNormKeys ? sh.norm : sh.full;  // staged (and normalised) tiles
    // Descriptors of stage 0: the stream's 64 token rows of the key tile
    // (K-major) and its value slices 4g .. 4g+3 with the ones tile (MN-major).
    // Stage s is s * kStageBytes further: the key descriptor's start address
    // moves by that much, and so does the value descriptor's, whose distance
    // to the ones tile (its leading byte offset field) shrinks by as much.
    // Both fields stay in range, so one multiply-add per stage moves them.
    const uint64_t dK0 = L::kmajor(smem_u32(sStage) + g * 64 * L::kRowBytes, 0);
    const uint64_t dV0 = L::values1(smem_u32(sStage) + kValueOff, aOnes, 4 * g);
    const uint64_t dDummy = L::kmajor(aOnes, 0);
    constexpr uint64_t kStep = kStageBytes >> 4;
    constexpr uint64_t kVStep = kStep - (kStep << 16);  // modulo 2^64
    // scores side: first tile of the next step to score, its stage and phase
    // parity; products side: stage of the first tile of the next step
    int s_tile = 0, s_stage = 0, p_stage = 0;
    uint32_t s_par = 0u;
    auto next_stage = [](int st) { return st + 1 == kStages ? 0 : st + 1; };
    // the tiles of the next step to score are staged (and normalised)
    auto scores_ready = [&]() -> bool {
      if (!warp_wait(sh, &ready_bar[s_stage], s_par)) return false;
      if (kLanes && s_tile + 1 < T) {
        const int s2 = next_stage(s_stage);
        return warp_wait(sh, &ready_bar[s2], s2 == 0 ? s_par ^ 1u : s_par);
      }
      return true;
    };
    // scores of the next step into buffer b: the latent queries (A) from
    // TMEM, the keys (B) from the staged tile; in the lanes layout lanes
    // 64-127 score the next tile. Past the end (`real` false) the ones tile
    // is scored: nothing reads it, its barrier only proves that the products
    // issued before it are complete.
    auto issue_s = [&](bool real, int b) {
      const uint32_t dS = gbase + 64 * b;
      if (!real) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) mma_ts_elect(dS, tQ + k * 8, L::adv(dDummy, 32 * k), idS, k > 0);
      } else {
        const uint64_t ka = dK0 + static_cast<uint64_t>(s_stage) * kStep;
        if (kLanes) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ts_masked_elect(dS, tQ + k * 8, L::adv(ka, 32 * k), idS, k > 0, kLo, kLo, kAll, kAll);
          if (s_tile + 1 < T) {
            const uint64_t kb = dK0 + static_cast<uint64_t>(next_stage(s_stage)) * kStep;
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_ts_masked_elect(dS, tQ + k * 8, L::adv(kb, 32 * k), idS, k > 0, kAll, kAll, kLo, kLo);
          }
        } else {
#pragma unroll
          for (int k = 0; k < D / 16; ++k) mma_ts_elect(dS, tQ + k * 8, L::adv(ka, 32 * k), idS, k > 0);
        }
        s_tile += kTps;
        s_stage += kTps;
        if (s_stage >= kStages) {
          s_stage -= kStages;
          s_par ^= 1u;
        }
      }
      mma_commit_elect(&sh.s_full[g][b]);
    };
    // O (+)= P [V | 1] of step j, P in buffer b
    auto issue_pv = [&](int j, int b) {
      const uint32_t aP = gbase + 64 * b + kColP;  // P over the buffer's second half
      const uint32_t first = j > 0 ? 1u : 0u;
      const uint64_t va = dV0 + static_cast<uint64_t>(p_stage) * kVStep;
      if (kLanes) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          mma_ts_masked_elect(dO, aP + i * 8, L::adv(va, i * 2 * L::kAtom), idO, i > 0 ? 1u : first, kLo, kLo, kAll,
                              kAll);
        if (kTps * j + 1 < T) {
          const uint64_t vb = dV0 + static_cast<uint64_t>(next_stage(p_stage)) * kVStep;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mma_ts_masked_elect(dO, aP + i * 8, L::adv(vb, i * 2 * L::kAtom), idO, i > 0 ? 1u : first, kAll, kAll,
                                kLo, kLo);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) mma_ts_elect(dO, aP + i * 8, L::adv(va, i * 2 * L::kAtom), idO, i > 0 ? 1u : first);
      }
      p_stage += kTps;
      if (p_stage >= kStages) p_stage -= kStages;
    };
    bool ok = U > 0 && warp_wait(sh, &sh.q_tmem[g], 0);
    tc_fence_after();
    // the first three score sets (past the end: proof-only sets)
#pragma unroll
    for (int b = 0; b < kBufs; ++b) {
      if (!ok) break;
      const bool real = b < U;
      if (real && !scores_ready()) {
        ok = false;
        break;
      }
      issue_s(real, b);
    }
    // Step j with buffer b: the products that read P, then at once the
    // scores of step j + 3 into the same buffer (U + 1 is the last one
    // issued). The stage of step j is released by the softmax warps once
    // these scores are done (they were issued after the products).
    auto step = [&](int j, int b, uint32_t par) -> bool {
      const bool more = j + kBufs <= U + 1, real = j + kBufs < U;
      if (real && !scores_ready()) return false;
      if (!warp_wait(sh, &sh.p_full[g][b], par)) return false;
      FLAREPP_TR(tr_on && lane == 0, kTrIssue + g, 3 * j);
      tc_fence_after();
      issue_pv(j, b);
      FLAREPP_TR(tr_on && lane == 0, kTrIssue + g, 3 * j + 1);
      if (more) issue_s(real, b);
      FLAREPP_TR(tr_on && lane == 0, kTrIssue + g, 3 * j + 2);
      return true;
    };
    uint32_t par = 0u;
    for (int j = 0; ok && j < U; j += kBufs, par ^= 1u) {
      ok = step(j, 0, par);
      if (ok && j + 1 < U) ok = step(j + 1, 1, par);
      if (ok && j + 2 < U) ok = step(j + 2, 2, par);
    }
    // every product of the stream is in before its accumulator is read, and
    // every MMA of this CTA completes before TMEM is released
    mma_commit_elect(&sh.o_full[g]);
    mma_commit_elect(&sh.drain);
    mbar_wait(&sh.drain, 0, sh.wait_limit);
  } else if (warp == kWarpNorm - 1 || warp == kWarpNorm || warp >= kWarpSoftmax + 8) {
    // ------------------------------------------- N0 of the synthesis keys
    // (rows 32p .. 32p+31 of every tile by warp 4, 5, 14, 15: one per SM
    // sub-partition)
    if (kNormKeys) {
      const int part = warp < kWarpSoftmax ? warp - (kWarpNorm - 1) : warp - (kWarpSoftmax + 6);  // 0, 1, 2, 3
      for (int t = 0; t < T; ++t) {
        if (!normalise_part<D, kStages>(sh, sStage, kStageBytes, t, part, lane)) break;
        FLAREPP_TR(tr_on && lane == 0, kTrNorm + part, t);
      }
    }
  } else if (warp >= kWarpSoftmax && warp < kWarpSoftmax + 8) {
    // ------------------------------------------------- softmax + epilogue
    const int tid = threadIdx.x - 32 * kWarpSoftmax;  // 0..255
    const int g = tid >> 7;                            // stream
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t gbase = tmem + lane_base + g * kGroupCols;
    const uint32_t tO = gbase + kColO;
    const int lanes_half = kLanes ? (row >> 6) : 0;  // the same in every lane of a warp
    const float c = rsqrtf((float)D) * kLog2e;
#ifdef FLAREPP_TRACE
    const bool tr_sm = tr_on && lane == 0 && (warp == kWarpSoftmax || warp == kWarpSoftmax + 4);
#endif
    // latent query row `row` of the staged block into the stream's Q columns
    // (lane = latent row, bf16 pairs)
    bool ok = wait_or_abort(sh, &sh.q_full, 0);
    if (ok) {
      uint32_t w[D / 2];
#pragma unroll
      for (int cc = 0; cc < D / 8; ++cc) {
        const uint4 v = *reinterpret_cast<const uint4*>(sQ + L::chunk_offset(row, cc));
        w[4 * cc] = v.x; w[4 * cc + 1] = v.y; w[4 * cc + 2] = v.z; w[4 * cc + 3] = v.w;
      }
      if (D == 32) tmem_st16(gbase + kColQ, *reinterpret_cast<uint32_t(*)[16]>(w));
      else tmem_st8(gbase + kColQ, *reinterpret_cast<uint32_t(*)[8]>(w));
      tmem_wait_st();
    }
    warp_arrive(&sh.q_tmem[g]);
    float r = -INFINITY, r_old = -INFINITY;  // the stream's reference (exp2 units)
    bool acc = false;                         // the accumulator holds products
    // One thread per stream releases the stage(s) of step j - 3 once the
    // scores of step j are done: the issuing thread issued them after the
    // products of step j - 3, the last reads of those stages by this stream.
    const bool rel_warp = (warp & 3) == (kWarpSoftmax & 3);  // one warp of each stream
    int rel_stage = 0;  // stage of the first tile of step j - 3
    // the stream's token columns in the last tile (every earlier step has 64)
    const int last_valid = min(kTile, n_end - (n_begin + (T - 1) * kTile)) - 64 * g;
    int b = 0;
    uint32_t par = 0u;  // phase parity of step j's barriers: (j / 3) & 1
    // Step j. kLast: the stream's last step, where the tile may be partial or
    // (lanes layout) absent; every other step is a full 64-column step with
    // no test of its columns.
    auto step = [&](int j, auto last_tag) -> bool {
      constexpr bool kLast = decltype(last_tag)::value;
      const uint32_t tS = gbase + 64 * b;
      if (!wait_or_abort(sh, &sh.s_full[g][b], par)) return false;
      FLAREPP_TR(tr_sm, kTrSoftmax + g, 2 * j);
      tc_fence_after();
      if (rel_warp && j >= kBufs) {
        mbar_arrive_if(&sh.empty[rel_stage], lane == 0);
        if (kLanes) mbar_arrive_if(&sh.empty[rel_stage + 1 == kStages ? 0 : rel_stage + 1], lane == 0 && kTps * (j - kBufs) + 1 < T);
        rel_stage += kTps;
        if (rel_stage >= kStages) rel_stage -= kStages;
      }
      bool moved = false, wrote = true;
      if (kLast) {
        const int t = kTps * j + lanes_half;
        const int valid = t + 1 < T ? 64 : (t < T ? last_valid : 0);  // the same in every lane of a warp
        if (valid > 0) {
          moved = softmax_step<true>(tS, min(valid, 64), j == 0, c, r, r_old);
        } else {
          wrote = false;
          if (t < T) zero_p(tS);  // no token in the stream's half of the last tile
        }
      } else {
        moved = softmax_step<false>(tS, 64, j == 0, c, r, r_old);
      }
      const int bp = b == 0 ? 2 : (b == 1 ? 0 : 1);  // buffer of step j + 2 and its phase
      const bool ok2 = finish_step<D>(sh, &sh.p_full[g][b], tO, r, r_old, acc, moved, &sh.s_full[g][bp],
                                      b == 0 ? par : par ^ 1u);
      FLAREPP_TR(tr_sm, kTrSoftmax + g, 2 * j + 1);
      if (wrote) acc = true;
      if (b == kBufs - 1) {
        b = 0;
        par ^= 1u;
      } else {
        ++b;
      }
      return ok2;
    };
    using Full = std::false_type;
    using Last = std::true_type;
    for (int j = 0; ok && j + 1 < U; ++j) ok = step(j, Full{});
    if (ok && U > 0) ok = step(U - 1, Last{});
    // every product of the stream is in before the accumulator is read
    if (ok && U > 0) ok = wait_or_abort(sh, &sh.o_full[g], 0);
    tc_fence_after();
    FLAREPP_TR(tr_on && tid == 0, kTrEpi, 0);

    // 1) each stream's (L, Z) into shared memory, stream e = 128 g + row
    //    (after the whole CTA's products are done: the scratch is the ring)
    float o[D];
    const float l = load_acc<D>(tO, o);
    if (ok) ok = wait_or_abort(sh, &sh.drain, 0);
    softmax_groups_sync();
    constexpr int kZs = D + 1;  // padded row stride
    float* scr_l = reinterpret_cast<float*>(sStage);  // [256]
    float* scr_z = scr_l + 256;                       // [256][D + 1]
    {
      const int e = 128 * g + row;
      const bool any = ok && acc && l > 0.f;  // a stream with no token never wrote its accumulator
      const float inv = any ? 1.f / l : 0.f;
      scr_l[e] = any ? (r + __log2f(l)) * kLn2 : -INFINITY;  // the accumulator is at reference r
#pragma unroll
      for (int d = 0; d < D; ++d) scr_z[e * kZs + d] = any ? o[d] * inv : 0.f;
    }
    softmax_groups_sync();

    // 2) the CTA's streams of a latent row merged (Appendix B.3 schedule):
    //    stream e holds latent row e & 127 (e & 63 in the lanes layout).
    //    With one split this is the final result; otherwise one partial per
    //    (latent row, split) and the last CTA of the head merges them.
    const int nwriters = kLanes ? 64 : 128;
    const int nent = 256 / nwriters;
    for (int e = tid; e < nwriters; e += 256) {
      const int latent = (kLanes ? 0 : qt * kTile) + e;
      if (latent >= p.M) continue;
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
      const float lse = dsum > 0.f ? lmax + __logf(dsum) : -INFINITY;
      if (p.splits == 1) {
        write_final<D, kKind>(p, bh, h, latent, u, lse);
      } else {
        const size_t prow = (((size_t)bh * p.qtiles + qt) * p.splits + split) * kTile + e;
        store_row<D>(p.part_z + prow * D, u);
        p.part_l[prow] = lse;
      }
    }
    if (p.splits > 1) {
      __threadfence();
      softmax_groups_sync();
      const size_t grp = (size_t)bh * p.qtiles + qt;
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
        // 3) the last CTA of the block merges the splits (Appendix B.3:
        //    L_max, d_s = exp(L_s - L_max), U = sum d_s Z_s, Z = U / d), with
        //    `tpr` threads per latent row sharing the splits
        const int rows = kLanes ? 64 : 128;
        const int tpr = 256 / rows;
        const int r_f = tid / tpr, part = tid % tpr;
        const int latent_f = (kLanes ? 0 : qt * kTile) + r_f;
        const size_t base = ((size_t)bh * p.qtiles + qt) * p.splits * kTile + r_f;
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
          const float invd = dsum > 0.f ? 1.f / dsum : 0.f;
#pragma unroll
          for (int d = 0; d < D; ++d) u[d] *= invd;
          write_final<D, kKind>(p, bh, h, latent_f, u, dsum > 0.f ? gmax + __logf(dsum) : -INFINITY);
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
  int fail_wait;       // test only: P barrier of stream 0, buffer 0 expects one arrival too many
};

// The decode's TMEM per stream, two layouts. Few route blocks per tile
// (M <= 128, kDbl): two 64-column score buffers (scores issued two steps
// ahead) and two accumulators that the stream's tiles use in turn, so that a
// tile's output goes out during the next tile without waiting for its last
// products. Otherwise: three score buffers (scores three steps ahead) and one
// accumulator; the output goes out at the next tile's first step.
template <bool kDbl>
struct DecLayout {
  static constexpr int kBufs = kDbl ? 2 : 3;
  static constexpr uint32_t kColO = kBufs * 64;
};
static_assert(DecLayout<true>::kColO + 2 * Layout<32>::kNo <= kGroupCols, "decode accumulators exceed a stream's columns");
static_assert(DecLayout<false>::kColO + Layout<32>::kNo <= kGroupCols, "decode accumulator exceeds a stream's columns");

// Token-tile ring depth of the decode kernel: a compile-time constant, so
// that the ring index and phase of a tile cost no division on the issuing
// threads. With Q and Z of M <= 512 routes resident it still fits.
constexpr int kDecodeStages = 12;
// At most this many heads' Q and Z per CTA, within this much shared memory.
constexpr int kDecodeHeads = 4;
constexpr int kDecodeSmemLimit = 220 * 1024;
template <int D>
__host__ __device__ constexpr int decode_smem_bytes(int M, int heads) {
  return 1024 + (2 * heads * ((M + kTile - 1) / kTile) + kDecodeStages + 1) * (int)Layout<D>::kTileBytes;
}
static_assert(decode_smem_bytes<32>(512, 1) <= kDecodeSmemLimit, "decode ring does not fit next to Q and Z");

template <int D, bool kDbl>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_z, const DecodeParams p) {
  using L = Layout<D>;
  constexpr int kDecBufs = DecLayout<kDbl>::kBufs;
  constexpr uint32_t kDecColO = DecLayout<kDbl>::kColO;
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
  // Schedule: stream g takes local tiles g, g + 2, g + 4, ... and runs over
  // all M routes of a tile in `nsub` steps of 64 routes, carrying its online
  // softmax over M from one step to the next, so its accumulator ends as a
  // whole output row. Step j of the stream: its (j / nsub)-th tile, routes
  // 64 (j % nsub) .. +63; counters advance without a division.
  const int nsub = (p.M + 63) / 64;
  // steps of stream g (a run-time index into an array would put it in local
  // memory)
  auto stream_steps = [&](int g) { return (T > g ? (T - g + 1) / 2 : 0) * nsub; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);  // a tile is read by one stream
    }
    mbar_init(&sh.q_full, 1);
    for (int g = 0; g < 2; ++g) {
      for (int b = 0; b < kDecBufs; ++b) {
        mbar_init(&sh.s_full[g][b], 1);
        mbar_init(&sh.p_full[g][b], 4 + (p.fail_wait && g == 0 && b == 0 ? 1 : 0));
      }
      mbar_init(&sh.o_full[g], 1);
    }
    mbar_init(&sh.drain, 2);
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
  } else if (warp == kWarpIssue || warp == kWarpIssue + 1) {
    // ------------------------------------------------ MMAs of stream g
    // Kept short as in the split kernel: unrolled over the three score
    // buffers, every ring stage, route block and descriptor moved by adds.
    const int g = warp - kWarpIssue;
    const uint32_t gbase = tmem + g * kGroupCols;
    const uint32_t aOnes = smem_u32(sOnes);
    const uint32_t idO = idesc_bf16(128, L::kNo, false, true);
    const uint32_t idS64 = idesc_bf16(128, 64, false, false);
    // the last route block holds M - 64 (nsub - 1) routes (a multiple of 16)
    const int wlast = p.M - 64 * (nsub - 1);
    const uint32_t idSlast = idesc_bf16(128, wlast, false, false);
    const int nsl_last = wlast / 16;
    // Descriptors: the K tile of ring stage s (K-major) is s tiles past
    // stage 0; routes 64b .. 64b+63 of the head at byte offset `hoff` are
    // hoff + 64b rows past the start of Q (K-major) and of Z (MN-major, with
    // the ones tile as its second column block, whose distance shrinks as
    // far as the start moves).
    const uint64_t dK0 = L::kmajor(smem_u32(sK), 0);
    const uint64_t dQ0 = L::kmajor(smem_u32(sQ), 0);
    const uint64_t dZ0 = L::values1(smem_u32(sZ), aOnes, 0);
    const uint64_t dDummy = L::kmajor(aOnes, 0);
    constexpr uint64_t kKStep = L::kTileBytes >> 4;
    constexpr uint64_t kBlk = (64 * L::kRowBytes) >> 4;
    constexpr uint64_t kZBlk = kBlk - (kBlk << 16);  // modulo 2^64
    auto q_head = [&](uint32_t hoff) { return dQ0 + (hoff >> 4); };
    auto z_head = [&](uint32_t hoff) { return dZ0 + (hoff >> 4) - (static_cast<uint64_t>(hoff >> 4) << 16); };
    const int U = stream_steps(g);
    // scores side: tile ts (local), block bs, its stage, phase parity and
    // descriptors; products side: tile tp, block bp, its stage and Z
    // descriptor
    int ts = g, bs = 0, stage_s = g;
    uint32_t par_s = 0u;
    uint64_t ks = dK0 + static_cast<uint64_t>(g) * kKStep, qs = q_head(head_slot(g) * head_bytes);
    int tp = g, bp = 0, stage_p = g;
    uint32_t dO = gbase + kDecColO;  // the accumulator of the products' tile (by the stream's tile parity)
    uint64_t zp = z_head(head_slot(g) * head_bytes);
    // scores of the next step into buffer b (past the end: the ones tile
    // against itself, a proof-only set)
    auto issue_s = [&](bool real, int b) -> bool {
      const uint32_t dS = gbase + 64 * b;
      if (real) {
        if (bs == 0 && !warp_wait(sh, &sh.full[stage_s], par_s)) return false;
        tc_fence_after();
        const uint32_t id = bs == nsub - 1 ? idSlast : idS64;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) mma_ss_elect(dS, L::adv(ks, 32 * k), L::adv(qs, 32 * k), id, k > 0);
        if (++bs == nsub) {
          bs = 0;
          ts += 2;
          stage_s += 2;
          if (stage_s >= stages) {
            stage_s -= stages;
            par_s ^= 1u;
          }
          ks = dK0 + static_cast<uint64_t>(stage_s) * kKStep;
          qs = q_head(head_slot(ts) * head_bytes);
        } else {
          qs += kBlk;
        }
      } else {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) mma_ss_elect(dS, L::adv(dDummy, 32 * k), L::adv(dDummy, 32 * k), idS64, k > 0);
      }
      mma_commit_elect(&sh.s_full[g][b]);
      return true;
    };
    // O (+)= P [Z | 1] over the route slices of the current block, P in
    // buffer b; after a tile's last block its stage is released and its
    // accumulator may be read out
    auto issue_pv = [&](int b) {
      const uint32_t aP = gbase + 64 * b + kColP;  // P over the buffer's second half
      const uint32_t first = bp > 0 ? 1u : 0u;
      if (bp < nsub - 1 || nsl_last == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) mma_ts_elect(dO, aP + i * 8, L::adv(zp, i * 2 * L::kAtom), idO, i > 0 ? 1u : first);
      } else {
        for (int i = 0; i < nsl_last; ++i)
          mma_ts_elect(dO, aP + i * 8, L::adv(zp, i * 2 * L::kAtom), idO, i > 0 ? 1u : first);
      }
      if (++bp == nsub) {
        mma_commit_elect(&sh.empty[stage_p]);
        mma_commit_elect(&sh.o_full[g]);
        bp = 0;
        tp += 2;
        if (kDbl) dO = dO == gbase + kDecColO ? gbase + kDecColO + L::kNo : gbase + kDecColO;
        stage_p += 2;
        if (stage_p >= stages) stage_p -= stages;
        zp = z_head(head_slot(tp) * head_bytes);
      } else {
        zp += kZBlk;
      }
    };
    bool ok = U > 0 && warp_wait(sh, &sh.q_full, 0);
    // the first two score sets
#pragma unroll
    for (int b = 0; b < kDecBufs; ++b) {
      if (!ok) break;
      ok = issue_s(b < U, b);
    }
    // step j with buffer b: the products, then the scores of step j + kDecBufs
    // into the same buffer (U + kDecBufs - 2 is the last one issued: proof-only
    // sets past the end)
    auto step = [&](int j, int b, uint32_t par) -> bool {
      if (!warp_wait(sh, &sh.p_full[g][b], par)) return false;
      FLAREPP_TR(tr_on && lane == 0, kTrIssue + g, 3 * j);
      tc_fence_after();
      issue_pv(b);
      FLAREPP_TR(tr_on && lane == 0, kTrIssue + g, 3 * j + 1);
      if (j + kDecBufs <= U + kDecBufs - 2 && !issue_s(j + kDecBufs < U, b)) return false;
      FLAREPP_TR(tr_on && lane == 0, kTrIssue + g, 3 * j + 2);
      return true;
    };
    uint32_t par = 0u;
    for (int j = 0; ok && j < U; j += kDecBufs, par ^= 1u) {
      ok = step(j, 0, par);
      if (ok && j + 1 < U) ok = step(j + 1, 1, par);
      if (kDecBufs == 3 && ok && j + 2 < U) ok = step(j + 2, 2, par);
    }
    mma_commit_elect(&sh.drain);
    mbar_wait(&sh.drain, 0, sh.wait_limit);
  } else if (warp >= kWarpSoftmax && warp < kWarpSoftmax + 8) {
    const int tid = threadIdx.x - 32 * kWarpSoftmax;  // 0..255
    const int g = tid >> 7;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t gbase = tmem + lane_base + g * kGroupCols;
    const float c = rsqrtf((float)D) * kLog2e;
    // the accumulator of the stream's i-th tile (two, by tile parity, in the
    // double layout)
    auto acc_of = [&](int i) { return gbase + kDecColO + (kDbl ? (i & 1) * L::kNo : 0u); };
#ifdef FLAREPP_TRACE
    const bool tr_sm = tr_on && lane == 0 && (warp == kWarpSoftmax || warp == kWarpSoftmax + 4);
#endif
    // out = O / rowsum of the accumulator, for local tile t (the i-th of the
    // stream), once the tile's products are done
    auto emit = [&](int i, int t) -> bool {
      const bool done = wait_or_abort(sh, &sh.o_full[g], i & 1);
      tc_fence_after();
      if (!done) return false;
      float z[D];
      const float l = load_acc<D>(acc_of(i), z);
      const int hs = head_slot(t);
      const int tok = (first + t - hs * n_tiles) * kTile + row;
      if (tok < p.N) {
        const float inv = 1.f / l;
#pragma unroll
        for (int d = 0; d < D; ++d) z[d] *= inv;
        store_row<D>(p.out + ((size_t)(h0 + hs) * p.N + tok) * D, z);
      }
      return true;
    };
    bool ok = true;
    float r = -INFINITY, r_old = -INFINITY;  // the reference of the current tile's stream over M
    bool acc = false;                         // the accumulator holds this tile's products
    const int wlast = p.M - 64 * (nsub - 1);  // routes of a tile's last block (16..64)
    const int ntiles = T > g ? (T - g + 1) / 2 : 0;
    int bf = 0, j = 0, i = 0;
    uint32_t par = 0u;  // phase parity of step j's barriers: (j / kDecBufs) & 1
    // Step j: route block b of the stream's i-th tile. kRagged: the last
    // block of a tile when M is not a multiple of 64 (its columns at or past
    // `wlast` count as absent); every other block has no test of its columns.
    auto step = [&](int b, auto ragged_tag) -> bool {
      constexpr bool kRagged = decltype(ragged_tag)::value;
      const uint32_t tS = gbase + 64 * bf;
      if (!wait_or_abort(sh, &sh.s_full[g][bf], par)) return false;
      FLAREPP_TR(tr_sm, kTrSoftmax + g, 2 * j);
      tc_fence_after();
      // a new tile (b == 0) starts a new stream over M: its reference comes
      // from its own first route block and its accumulator starts empty
      if (b == 0) acc = false;
      const bool moved = softmax_step<kRagged>(tS, kRagged ? wlast : 64, b == 0, c, r, r_old);
      // The previous tile's output goes out before the products that
      // overwrite its accumulator: in the double layout at this tile's last
      // step (its own last products were issued a whole tile ago), otherwise
      // at this tile's first step.
      if (b == (kDbl ? nsub - 1 : 0) && i > 0 && !emit(i - 1, g + 2 * (i - 1))) return false;
      // proof of the previous products: the scores issued after them, those
      // of step j + kDecBufs - 1
      const int bp = kDbl ? (bf ^ 1) : (bf == 0 ? 2 : (bf == 1 ? 0 : 1));
      const bool ok2 = finish_step<D>(sh, &sh.p_full[g][bf], acc_of(i), r, r_old, acc, moved,
                                      &sh.s_full[g][bp], bf == 0 ? par : par ^ 1u);
      FLAREPP_TR(tr_sm, kTrSoftmax + g, 2 * j + 1);
      acc = true;
      if (bf == kDecBufs - 1) {
        bf = 0;
        par ^= 1u;
      } else {
        ++bf;
      }
      ++j;
      return ok2;
    };
    using Full = std::false_type;
    using Ragged = std::true_type;
    for (i = 0; ok && i < ntiles; ++i) {
      for (int b = 0; ok && b + 1 < nsub; ++b) ok = step(b, Full{});
      if (ok) ok = wlast < 64 ? step(nsub - 1, Ragged{}) : step(nsub - 1, Full{});
    }
    // the stream's last tile
    if (ok && ntiles > 0) emit(ntiles - 1, g + 2 * (ntiles - 1));
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
  return 1024 + 2 * (size_t)Layout<D>::kTileBytes + split_stages<D, kKind>() * stage;
}

template <int D>
size_t decode_smem(int M, int heads) {
  return (size_t)decode_smem_bytes<D>(M, heads);
}

template <int D, int kKind, bool kLanes>
cudaError_t launch_split_layout(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                const SplitParams& a, dim3 grid, cudaStream_t stream, const char* what,
                                const char** failed) {
  const size_t smem = split_smem<D, kKind>();
  *failed = "cudaFuncSetAttribute(split_kernel)";
  cudaError_t e =
      cudaFuncSetAttribute(split_kernel<D, kKind, kLanes>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  split_kernel<D, kKind, kLanes><<<grid, kThreads, smem, stream>>>(mq, mk, mv, a);
  *failed = what;
  return cudaGetLastError();
}

// M <= 64 takes the lanes layout (two token tiles per step)
template <int D, int kKind>
cudaError_t launch_split(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const SplitParams& a,
                         dim3 grid, cudaStream_t stream, const char* what, const char** failed) {
  return a.M <= 64 ? launch_split_layout<D, kKind, true>(mq, mk, mv, a, grid, stream, what, failed)
                   : launch_split_layout<D, kKind, false>(mq, mk, mv, a, grid, stream, what, failed);
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
    // two route blocks or fewer per tile: the double-accumulator layout
    auto kernel = pr.M <= 128 ? decode_kernel<D, true> : decode_kernel<D, false>;
    if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return e;
    kernel<<<pl.decode_ctas, kThreads, smem, stream>>>(m_k, m_qdec, m_zdec, d);
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
  // one CTA per block of 128 latent rows (M <= 64: one block, its rows
  // repeated in TMEM lanes 64-127)
  pl.tiles = M <= 64 ? 1 : (M + tc::kTile - 1) / tc::kTile;
  pl.qgroups = pl.tiles;
  pl.streams = 1;  // the token streams of a CTA are merged before its partial is written
  // token tiles per split: at least 4 when the sequence allows
  const int splits = tc::choose_splits(BH * pl.qgroups, n_tiles, std::max(1, sms), 4, 12, forced_splits);
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
