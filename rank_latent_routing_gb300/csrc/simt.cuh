// FP32 CUDA-core kernels of the FLARE++ mixer forward.
//
// These carry the fp32 verification build (every product and softmax in
// fp32 on the CUDA cores) with the same decomposition as the tensor-core
// path: split-N passes whose partial results are merged by the last CTA to
// arrive (FLARE++ Appendix B.3 schedule, eq. 29-33, applied across CTAs of one
// GPU instead of across ranks), then a decode pass.
#pragma once

#include "common.cuh"

namespace flarepp {
namespace simt {

constexpr int kRows = 128;   // latent rows per CTA, one per thread
constexpr int kTile = 32;    // tokens staged in shared memory per step

template <typename T>
struct SplitArgs {
  const T* keys;      // [BH][N][D]
  const T* values;    // [BH][N][D]; unused when the keys serve as values
  const T* queries;   // [H][M][D] (q_by_head) or [BH][M][D]
  const T* qf;        // gated passes only: Qf [H][M][D]
  const float* gate;  // gated passes only: g [H]
  int q_by_head;
  int H, N, M, tiles, splits, split_len;
  Partials part;
  T* out;             // gated: Q [BH][M][D]; encode: Z [BH][M][D]
  float* dbg_a;       // gated: Qd fp32; encode: Z fp32 (as rounded); may be null
  float* dbg_b;       // gated: Q fp32 (as rounded); encode: L fp32; may be null
  float* dbg_c;       // gated: L of the synthesis softmax (natural log); may be null
};

// One CTA = one (split, 128-row tile of latents, batch*head). Each thread
// owns one latent row: it scores the staged tokens, keeps a running max and
// sum in the log2 domain and accumulates its unnormalised output row.
template <typename T, int D, int kKind>
__global__ void __launch_bounds__(kRows) split_kernel(const SplitArgs<T> a) {
  constexpr bool kNormKeys = pass_normalises_keys(kKind);
  constexpr bool kSepValues = pass_separate_values(kKind);
  const int s = blockIdx.x, tile = blockIdx.y, bh = blockIdx.z;
  const int h = bh % a.H;
  const int tid = threadIdx.x;
  const int m = tile * kRows + tid;
  const bool valid = m < a.M;

  __shared__ float ks[kTile][D];
  __shared__ float vs[kSepValues ? kTile : 1][D];
  __shared__ int s_last;

  // queries pre-scaled by 1/sqrt(D) * log2(e): scores come out in log2 units
  float q[D];
  const float qscale = rsqrtf((float)D) * kLog2e;
  if (valid) {
    const T* qrow = a.queries + ((size_t)(a.q_by_head ? h : bh) * a.M + m) * D;
#pragma unroll
    for (int d = 0; d < D; ++d) q[d] = to_f32(qrow[d]) * qscale;
  } else {
#pragma unroll
    for (int d = 0; d < D; ++d) q[d] = 0.f;
  }

  float mrun = -INFINITY, lrun = 0.f, o[D];
#pragma unroll
  for (int d = 0; d < D; ++d) o[d] = 0.f;

  const size_t base = (size_t)bh * a.N * D;
  const int n_begin = s * a.split_len;
  const int n_end = min(a.N, n_begin + a.split_len);
  for (int n0 = n_begin; n0 < n_end; n0 += kTile) {
    const int cnt = min(kTile, n_end - n0);
    __syncthreads();
    // rows past the split's end are zero-filled: their weights are 0, and
    // 0 * (stale shared memory) could be NaN
    for (int e = tid; e < kTile * D; e += kRows) {
      const bool in = e < cnt * D;
      ks[e / D][e % D] = in ? to_f32(a.keys[base + (size_t)n0 * D + e]) : 0.f;
      if constexpr (kSepValues) vs[e / D][e % D] = in ? to_f32(a.values[base + (size_t)n0 * D + e]) : 0.f;
    }
    if (kNormKeys) {
      // N0 of the synthesis keys (eq. 5): one thread per staged token row
      __syncthreads();
      if (tid < cnt) {
        float ss = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) ss += ks[tid][d] * ks[tid][d];
        const float r = rsqrtf(ss / (float)D + kEps);
#pragma unroll
        for (int d = 0; d < D; ++d) ks[tid][d] *= r;
      }
    }
    __syncthreads();
    if (!valid) continue;
    float sc[kTile];
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < kTile; ++j) {
      float acc = 0.f;
#pragma unroll
      for (int d = 0; d < D; ++d) acc = fmaf(q[d], ks[j][d], acc);
      sc[j] = j < cnt ? acc : -INFINITY;
      tmax = fmaxf(tmax, sc[j]);
    }
    const float mnew = fmaxf(mrun, tmax);
    const float corr = exp2f(mrun - mnew);
    lrun *= corr;
#pragma unroll
    for (int d = 0; d < D; ++d) o[d] *= corr;
#pragma unroll
    for (int j = 0; j < kTile; ++j) {
      const float p = exp2f(sc[j] - mnew);
      lrun += p;
      if constexpr (!kSepValues) {
        // the synthesis pass shares its normalised keys as values (eq. 19);
        // re-read them so the compiler does not hold the whole tile in registers
        const volatile float* kv = ks[j];
#pragma unroll
        for (int d = 0; d < D; ++d) o[d] = fmaf(p, kv[d], o[d]);
      } else {
#pragma unroll
        for (int d = 0; d < D; ++d) o[d] = fmaf(p, vs[j][d], o[d]);
      }
    }
    mrun = mnew;
  }

  // this split's (Z_s, L_s); an empty split gives Z_s = 0, L_s = -inf
  const size_t prow = (((size_t)bh * a.tiles + tile) * a.splits + s) * kRows + tid;
  if (valid) {
    float z[D];
    const float inv = lrun > 0.f ? 1.f / lrun : 0.f;
#pragma unroll
    for (int d = 0; d < D; ++d) z[d] = o[d] * inv;
    store_row<D>(a.part.z + prow * D, z);
    a.part.l[prow] = lrun > 0.f ? (mrun + log2f(lrun)) * kLn2 : -INFINITY;
  }
  __threadfence();
  __syncthreads();
  unsigned* counter = a.part.counters + (size_t)bh * a.tiles + tile;
  if (tid == 0) s_last = atomicAdd(counter, 1u) == (unsigned)(a.splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) *counter = 0u;  // ready for the next call
  if (!valid) return;

  // merge the splits: L_max, d_s = exp(L_s - L_max), U = sum d_s Z_s, Z = U/d
  const size_t p0 = (((size_t)bh * a.tiles + tile) * a.splits) * kRows + tid;
  float lmax = -INFINITY;
  for (int t = 0; t < a.splits; ++t) lmax = fmaxf(lmax, __ldcg(a.part.l + p0 + (size_t)t * kRows));
  float u[D], dsum = 0.f;
#pragma unroll
  for (int d = 0; d < D; ++d) u[d] = 0.f;
  for (int t = 0; t < a.splits; ++t) {
    const size_t r = p0 + (size_t)t * kRows;
    const float lt = __ldcg(a.part.l + r);
    if (lt == -INFINITY) continue;
    const float w = expf(lt - lmax);
    dsum += w;
#pragma unroll
    for (int d = 0; d < D; ++d) u[d] = fmaf(w, __ldcg(a.part.z + r * D + d), u[d]);
  }
  const float invd = 1.f / dsum;
#pragma unroll
  for (int d = 0; d < D; ++d) u[d] *= invd;
  const size_t orow = (size_t)bh * a.M + m;
  if (pass_gated(kKind)) {
    // gate (eq. 7): Q = N0(Qf) + g * Qd, evaluated in fp32, then cast
    const T* qfrow = a.qf + ((size_t)h * a.M + m) * D;
    float f[D], ss = 0.f;
#pragma unroll
    for (int d = 0; d < D; ++d) { f[d] = to_f32(qfrow[d]); ss += f[d] * f[d]; }
    const float r = rsqrtf(ss / (float)D + kEps);
    const float g = a.gate[h];
    float qo[D];
#pragma unroll
    for (int d = 0; d < D; ++d) qo[d] = fmaf(g, u[d], f[d] * r);
    if (a.dbg_a) store_row<D>(a.dbg_a + orow * D, u);
    if (a.dbg_c) a.dbg_c[orow] = lmax + logf(dsum);
#pragma unroll
    for (int d = 0; d < D; ++d) {
      a.out[orow * D + d] = from_f32<T>(qo[d]);
      if (a.dbg_b) a.dbg_b[orow * D + d] = round_as<T>(qo[d]);
    }
  } else {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      a.out[orow * D + d] = from_f32<T>(u[d]);
      if (a.dbg_a) a.dbg_a[orow * D + d] = round_as<T>(u[d]);
    }
    if (a.dbg_b) a.dbg_b[orow] = lmax + logf(dsum);
  }
}

template <typename T>
struct DecodeArgs {
  const T* keys;  // [BH][N][D]
  const T* q;     // [H][M][D] (q_by_head) or [BH][M][D]
  const T* z;     // [BH][M][D]
  T* out;         // [BH][N][D]
  int N, M, H, q_by_head;
};

constexpr int kDecodeTokens = 128;  // tokens per CTA, one per thread
constexpr int kDecodeChunk = 32;    // routes scored per online-softmax step

// One CTA = 128 tokens of one (batch, head). Q and Z of the head sit in
// shared memory (fp32); each thread runs the softmax over the M routes for
// its token and accumulates its output row.
template <typename T, int D>
__global__ void __launch_bounds__(kDecodeTokens) decode_kernel(const DecodeArgs<T> a) {
  extern __shared__ float smem[];
  float* qs = smem;              // [M][D], scaled by 1/sqrt(D)*log2(e)
  float* zs = smem + a.M * D;    // [M][D]
  const int bh = blockIdx.y;
  const int tid = threadIdx.x;
  const float qscale = rsqrtf((float)D) * kLog2e;
  const size_t lbase = (size_t)bh * a.M * D;
  const size_t qbase = (size_t)(a.q_by_head ? bh % a.H : bh) * a.M * D;
  for (int e = tid; e < a.M * D; e += kDecodeTokens) {
    qs[e] = to_f32(a.q[qbase + e]) * qscale;
    zs[e] = to_f32(a.z[lbase + e]);
  }
  __syncthreads();
  const int n = blockIdx.x * kDecodeTokens + tid;
  if (n >= a.N) return;
  float k[D];
  load_row<D>(a.keys + ((size_t)bh * a.N + n) * D, k);
  float mrun = -INFINITY, lrun = 0.f, y[D];
#pragma unroll
  for (int d = 0; d < D; ++d) y[d] = 0.f;
  for (int m0 = 0; m0 < a.M; m0 += kDecodeChunk) {
    float sc[kDecodeChunk];
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < kDecodeChunk; ++j) {
      const int mm = m0 + j;
      float acc = 0.f;
      if (mm < a.M) {
#pragma unroll
        for (int d = 0; d < D; ++d) acc = fmaf(k[d], qs[mm * D + d], acc);
      }
      sc[j] = mm < a.M ? acc : -INFINITY;
      tmax = fmaxf(tmax, sc[j]);
    }
    const float mnew = fmaxf(mrun, tmax);
    const float corr = exp2f(mrun - mnew);
    lrun *= corr;
#pragma unroll
    for (int d = 0; d < D; ++d) y[d] *= corr;
#pragma unroll
    for (int j = 0; j < kDecodeChunk; ++j) {
      const int mm = m0 + j;
      if (mm >= a.M) break;
      const float p = exp2f(sc[j] - mnew);
      lrun += p;
#pragma unroll
      for (int d = 0; d < D; ++d) y[d] = fmaf(p, zs[mm * D + d], y[d]);
    }
    mrun = mnew;
  }
  const float inv = 1.f / lrun;
#pragma unroll
  for (int d = 0; d < D; ++d) y[d] *= inv;
  store_row<D>(a.out + ((size_t)bh * a.N + n) * D, y);
}

}  // namespace simt
}  // namespace flarepp
