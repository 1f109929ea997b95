// Backward pass of the FLARE++ mixer (the training direction), fp32 math on
// the CUDA cores for bf16 or fp32 inputs.
//
// Each of the three attention calls out = softmax(s q k^T) v is
// differentiated with the local backward of the FLARE++ paper (Appendix B.5
// eq. 46-49, one shard, merged log-normaliser L, no cotangent on L):
//   P = exp(S - L),  c = <dout, out> per row,  dS = P o (dout v^T - c),
//   dv = P^T dout,   dk = s dS^T q,             dq = s dS k.
// The gate and the two N0s follow by the chain rule. The passes:
//
//   recompute  the forward's synthesis and encode (SIMT kernels), keeping
//              Qd, Q (as rounded), Z (as rounded), L_syn and L_enc;
//   dec-token  one thread per token: the decode softmax over M again, its
//              log-normaliser and c_n = <dY_n, Y_n> = sum_m P dY.Z_m, and the
//              token's dK from the decode;
//   dec-latent one thread per latent route, token splits: dZ_m and the
//              decode's dQ_m; merged over the splits, then c_m = <dZ_m, Z_m>;
//   enc-token  one thread per token: dV_n and the encode's dK_n;
//   enc-latent one thread per route: the encode's dQ_m; the merge adds the
//              decode's, then the gate (dQd = g dQ, dg = <dQ, Qd>) and N0 of
//              Qf, and c_m = <dQd_m, Qd_m> for the synthesis;
//   syn-token  one thread per token: dKt_n as keys and values, then N0's
//              backward to dKs_raw;
//   syn-latent one thread per route: dQseed_m;
//   reduce     the per-head parameters' gradients summed over the batch in a
//              fixed order (deterministic).
//
// Token-major kernels hold the head's M x D latent tensors in shared memory;
// latent-major kernels stage 32 tokens at a time, like the forward's CUDA-core
// kernels. Every reduction has a fixed order, so results are bitwise
// repeatable.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "simt.cuh"

namespace flarepp {
namespace bwd {

constexpr int kRows = 128;     // threads per block: one token or one latent each
constexpr int kTileTok = 32;   // tokens staged per step in the latent-major kernels

template <int D>
__device__ __forceinline__ float dot(const float* a, const float* b) {
  float acc = 0.f;
#pragma unroll
  for (int d = 0; d < D; ++d) acc = fmaf(a[d], b[d], acc);
  return acc;
}

template <typename T, int D>
__device__ __forceinline__ void load_t(const T* p, float* out) {
#pragma unroll
  for (int d = 0; d < D; ++d) out[d] = to_f32(p[d]);
}

// ------------------------------------------------------------ dec-token
// Token n of head bh: the decode softmax over the M routes (queries K_n, keys
// Q, values Z), its log2-normaliser, c_n = sum_m P_nm <dY_n, Z_m>, and the
// decode's contribution to dK_n.
template <typename T, int D>
__global__ void __launch_bounds__(kRows)
    dec_token_kernel(const T* __restrict__ K, const T* __restrict__ dY, const float* __restrict__ Q,
                     const float* __restrict__ Z, int N, int M, float* __restrict__ dK,
                     float* __restrict__ Ldec, float* __restrict__ cdec) {
  extern __shared__ float sm[];
  float* qs = sm;          // [M][D]
  float* zs = sm + M * D;  // [M][D]
  const int bh = blockIdx.y;
  for (int e = threadIdx.x; e < M * D; e += kRows) {
    qs[e] = Q[(size_t)bh * M * D + e];
    zs[e] = Z[(size_t)bh * M * D + e];
  }
  __syncthreads();
  const int n = blockIdx.x * kRows + threadIdx.x;
  if (n >= N) return;
  const size_t row = ((size_t)bh * N + n) * D;
  float k[D], dy[D];
  load_t<T, D>(K + row, k);
  load_t<T, D>(dY + row, dy);
  const float c2 = rsqrtf((float)D) * kLog2e;  // scores in log2 units
  float mx = -INFINITY, sum = 0.f;
  for (int m = 0; m < M; ++m) {
    const float sc = c2 * dot<D>(k, qs + m * D);
    const float mn = fmaxf(mx, sc);
    sum = sum * exp2f(mx - mn) + exp2f(sc - mn);
    mx = mn;
  }
  const float L2 = mx + log2f(sum);
  float c = 0.f;
  for (int m = 0; m < M; ++m) {
    const float p = exp2f(c2 * dot<D>(k, qs + m * D) - L2);
    c = fmaf(p, dot<D>(dy, zs + m * D), c);
  }
  const float s = rsqrtf((float)D);
  float dk[D];
#pragma unroll
  for (int d = 0; d < D; ++d) dk[d] = 0.f;
  for (int m = 0; m < M; ++m) {
    const float* q = qs + m * D;
    const float p = exp2f(c2 * dot<D>(k, q) - L2);
    const float ds = p * (dot<D>(dy, zs + m * D) - c);
#pragma unroll
    for (int d = 0; d < D; ++d) dk[d] = fmaf(s * ds, q[d], dk[d]);
  }
  store_row<D>(dK + row, dk);
  Ldec[(size_t)bh * N + n] = L2;
  cdec[(size_t)bh * N + n] = c;
}

// ----------------------------------------------------------- enc-token
// Token n: the encode's gradients of its key and value rows, dV_n and the
// encode part of dK_n (added to the decode part already in dK).
template <typename T, int D>
__global__ void __launch_bounds__(kRows)
    enc_token_kernel(const T* __restrict__ K, const T* __restrict__ V, const float* __restrict__ Q,
                     const float* __restrict__ dZ, const float* __restrict__ Lenc,
                     const float* __restrict__ cenc, int N, int M, float* __restrict__ dK,
                     float* __restrict__ dV) {
  extern __shared__ float sm[];
  float* qs = sm;               // [M][D]
  float* dzs = sm + M * D;      // [M][D]
  float* l2s = sm + 2 * M * D;  // [M] log2-normalisers
  float* cs = l2s + M;          // [M]
  const int bh = blockIdx.y;
  for (int e = threadIdx.x; e < M * D; e += kRows) {
    qs[e] = Q[(size_t)bh * M * D + e];
    dzs[e] = dZ[(size_t)bh * M * D + e];
  }
  for (int m = threadIdx.x; m < M; m += kRows) {
    l2s[m] = Lenc[(size_t)bh * M + m] * kLog2e;
    cs[m] = cenc[(size_t)bh * M + m];
  }
  __syncthreads();
  const int n = blockIdx.x * kRows + threadIdx.x;
  if (n >= N) return;
  const size_t row = ((size_t)bh * N + n) * D;
  float k[D], v[D], dk[D], dv[D];
  load_t<T, D>(K + row, k);
  load_t<T, D>(V + row, v);
  load_row<D>(dK + row, dk);
#pragma unroll
  for (int d = 0; d < D; ++d) dv[d] = 0.f;
  const float c2 = rsqrtf((float)D) * kLog2e;
  const float s = rsqrtf((float)D);
  for (int m = 0; m < M; ++m) {
    const float* q = qs + m * D;
    const float* dz = dzs + m * D;
    const float p = exp2f(c2 * dot<D>(k, q) - l2s[m]);
    const float ds = p * (dot<D>(dz, v) - cs[m]);
#pragma unroll
    for (int d = 0; d < D; ++d) {
      dv[d] = fmaf(p, dz[d], dv[d]);
      dk[d] = fmaf(s * ds, q[d], dk[d]);
    }
  }
  store_row<D>(dK + row, dk);
  store_row<D>(dV + row, dv);
}

// ----------------------------------------------------------- syn-token
// Token n: the synthesis keys Kt_n = N0(Ks_raw_n) serve as keys and values;
// their gradient from both roles, then N0's backward to dKs_raw_n.
template <typename T, int D>
__global__ void __launch_bounds__(kRows)
    syn_token_kernel(const T* __restrict__ Ks, const T* __restrict__ Qseed, const float* __restrict__ dQd,
                     const float* __restrict__ Lsyn, const float* __restrict__ csyn, int N, int M, int H,
                     float* __restrict__ dKs) {
  extern __shared__ float sm[];
  float* qs = sm;               // [M][D] seeds of the head
  float* dqs = sm + M * D;      // [M][D]
  float* l2s = sm + 2 * M * D;  // [M]
  float* cs = l2s + M;          // [M]
  const int bh = blockIdx.y;
  const int h = bh % H;
  for (int e = threadIdx.x; e < M * D; e += kRows) {
    qs[e] = to_f32(Qseed[(size_t)h * M * D + e]);
    dqs[e] = dQd[(size_t)bh * M * D + e];
  }
  for (int m = threadIdx.x; m < M; m += kRows) {
    l2s[m] = Lsyn[(size_t)bh * M + m] * kLog2e;
    cs[m] = csyn[(size_t)bh * M + m];
  }
  __syncthreads();
  const int n = blockIdx.x * kRows + threadIdx.x;
  if (n >= N) return;
  const size_t row = ((size_t)bh * N + n) * D;
  float kt[D], g[D];
  load_t<T, D>(Ks + row, kt);
  const float r = rsqrtf(dot<D>(kt, kt) / (float)D + kEps);
#pragma unroll
  for (int d = 0; d < D; ++d) {
    kt[d] *= r;
    g[d] = 0.f;
  }
  const float c2 = rsqrtf((float)D) * kLog2e;
  const float s = rsqrtf((float)D);
  for (int m = 0; m < M; ++m) {
    const float* q = qs + m * D;
    const float* dq = dqs + m * D;
    const float p = exp2f(c2 * dot<D>(kt, q) - l2s[m]);
    const float ds = p * (dot<D>(dq, kt) - cs[m]);
#pragma unroll
    for (int d = 0; d < D; ++d) g[d] = fmaf(p, dq[d], fmaf(s * ds, q[d], g[d]));
  }
  // N0 backward: dx = r (g - kt <g, kt> / D)
  const float proj = dot<D>(g, kt) / (float)D;
#pragma unroll
  for (int d = 0; d < D; ++d) g[d] = r * (g[d] - kt[d] * proj);
  store_row<D>(dKs + row, g);
}

// -------------------------------------------------------- latent-major
// One thread per latent route m of a 128-route tile, over one token split;
// the split's sums go to partial buffers, summed over the splits afterwards.
//   kLatDec  the decode's value and key gradients of route m:
//            dZ_m = sum_n P_nm dY_n,  dQ_m = s sum_n dS_nm K_n
//   kLatEnc  the encode's query gradient dQ_m = s sum_n dS_mn K_n
//   kLatSyn  the synthesis' seed gradient dQseed_m = s sum_n dS_mn Kt_n
enum : int { kLatDec = 0, kLatEnc = 1, kLatSyn = 2 };

template <typename T>
struct LatArgs {
  const T* keys;       // [BH][N][D]: K (decode, encode) or Ks_raw (synthesis)
  const T* vals;       // [BH][N][D]: dY (decode) or V (encode); unused by the synthesis
  const float* tok_l;  // decode: per-token log2-normaliser [BH][N]
  const float* tok_c;  // decode: per-token c_n [BH][N]
  const float* lat_q;  // decode, encode: routing queries Q [BH][M][D]
  const T* seeds;      // synthesis: Qseed [H][M][D]
  const float* lat_o;  // decode: Z; encode: dZ; synthesis: dQd ([BH][M][D])
  const float* lat_l;  // encode, synthesis: natural log-normaliser [BH][M]
  const float* lat_c;  // encode, synthesis: c_m [BH][M]
  int H, N, M, tiles, splits, split_len;
  float* part1;        // [BH][tiles][splits][128][D]
  float* part2;        // decode only, same layout
};

template <typename T, int D, int kMode>
__global__ void __launch_bounds__(kRows) latent_kernel(const LatArgs<T> a) {
  const int split = blockIdx.x, tile = blockIdx.y, bh = blockIdx.z;
  const int h = bh % a.H;
  const int tid = threadIdx.x;
  const int m = tile * kRows + tid;
  const bool valid = m < a.M;
  __shared__ float ks[kTileTok][D];
  __shared__ float vs[kMode == kLatSyn ? 1 : kTileTok][D];
  __shared__ float tl[kTileTok], tc[kTileTok];

  float q[D], o[D];
  float l2 = 0.f, c = 0.f;
  if (valid) {
    if (kMode == kLatSyn) load_t<T, D>(a.seeds + ((size_t)h * a.M + m) * D, q);
    else load_row<D>(a.lat_q + ((size_t)bh * a.M + m) * D, q);
    load_row<D>(a.lat_o + ((size_t)bh * a.M + m) * D, o);
    if (kMode != kLatDec) {
      l2 = a.lat_l[(size_t)bh * a.M + m] * kLog2e;
      c = a.lat_c[(size_t)bh * a.M + m];
    }
  } else {
#pragma unroll
    for (int d = 0; d < D; ++d) q[d] = o[d] = 0.f;
  }
  float acc1[D], acc2[D];
#pragma unroll
  for (int d = 0; d < D; ++d) acc1[d] = acc2[d] = 0.f;
  const float c2 = rsqrtf((float)D) * kLog2e;
  const float s = rsqrtf((float)D);
  const size_t base = (size_t)bh * a.N * D;
  const int n_begin = split * a.split_len;
  const int n_end = min(a.N, n_begin + a.split_len);
  for (int n0 = n_begin; n0 < n_end; n0 += kTileTok) {
    const int cnt = min(kTileTok, n_end - n0);
    __syncthreads();
    for (int e = tid; e < kTileTok * D; e += kRows) {
      const bool in = e < cnt * D;
      ks[e / D][e % D] = in ? to_f32(a.keys[base + (size_t)n0 * D + e]) : 0.f;
      if constexpr (kMode != kLatSyn) vs[e / D][e % D] = in ? to_f32(a.vals[base + (size_t)n0 * D + e]) : 0.f;
    }
    if (kMode == kLatDec && tid < kTileTok) {
      tl[tid] = tid < cnt ? a.tok_l[(size_t)bh * a.N + n0 + tid] : 0.f;
      tc[tid] = tid < cnt ? a.tok_c[(size_t)bh * a.N + n0 + tid] : 0.f;
    }
    if (kMode == kLatSyn) {
      // N0 of the staged synthesis keys (eq. 5), one thread per token row
      __syncthreads();
      if (tid < cnt) {
        float ss = 0.f;
#pragma unroll
        for (int d = 0; d < D; ++d) ss = fmaf(ks[tid][d], ks[tid][d], ss);
        const float r = rsqrtf(ss / (float)D + kEps);
#pragma unroll
        for (int d = 0; d < D; ++d) ks[tid][d] *= r;
      }
    }
    __syncthreads();
    if (!valid) continue;
    for (int j = 0; j < cnt; ++j) {
      const float* kn = ks[j];
      if (kMode == kLatDec) {
        // route m as the key of token n's decode softmax
        const float p = exp2f(c2 * dot<D>(kn, q) - tl[j]);
        const float ds = p * (dot<D>(vs[j], o) - tc[j]);
#pragma unroll
        for (int d = 0; d < D; ++d) {
          acc1[d] = fmaf(p, vs[j][d], acc1[d]);
          acc2[d] = fmaf(s * ds, kn[d], acc2[d]);
        }
      } else {
        const float p = exp2f(c2 * dot<D>(q, kn) - l2);
        const float* vn = kMode == kLatSyn ? kn : vs[j];
        const float ds = p * (dot<D>(o, vn) - c);
#pragma unroll
        for (int d = 0; d < D; ++d) acc1[d] = fmaf(s * ds, kn[d], acc1[d]);
      }
    }
  }
  if (!valid) return;
  const size_t prow = (((size_t)bh * a.tiles + tile) * a.splits + split) * kRows + tid;
  store_row<D>(a.part1 + prow * D, acc1);
  if (kMode == kLatDec) store_row<D>(a.part2 + prow * D, acc2);
}

// The sum over splits of one latent route's partial rows.
template <int D>
__device__ __forceinline__ void sum_splits(const float* part, int bh, int tiles, int splits, int m, float* out) {
  const int tile = m / kRows, r = m % kRows;
#pragma unroll
  for (int d = 0; d < D; ++d) out[d] = 0.f;
  for (int sp = 0; sp < splits; ++sp) {
    float x[D];
    load_row<D>(part + ((((size_t)bh * tiles + tile) * splits + sp) * kRows + r) * D, x);
#pragma unroll
    for (int d = 0; d < D; ++d) out[d] += x[d];
  }
}

struct MergeArgs {
  int H, M, tiles, splits;
  const float* part1;
  const float* part2;
  const float* Z;       // decode: routes' values
  const float* Qd;      // encode: synthesis output
  const void* Qf;       // encode: fixed queries [H][M][D] (model dtype)
  const float* gate;    // encode: [H]
  float* dZ;            // decode: out
  float* dQ;            // decode: out (decode part); encode: in, then the total
  float* c_out;         // decode: c of the encode; encode: c of the synthesis
  float* dQd;           // encode: out
  float* dg_part;       // encode: <dQ, Qd> per (bh, m)
  float* dqf_part;      // encode: N0 backward of Qf per (bh, m)
  float* dqs_part;      // synthesis: seed gradient per (bh, m)
};

// One thread per (bh, m): the split sums and each pass's epilogue.
template <typename T, int D, int kMode>
__global__ void merge_kernel(const MergeArgs a, int BH) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= BH * a.M) return;
  const int bh = i / a.M, m = i % a.M, h = bh % a.H;
  const size_t row = ((size_t)bh * a.M + m) * D;
  float x[D];
  sum_splits<D>(a.part1, bh, a.tiles, a.splits, m, x);
  if (kMode == kLatDec) {
    float z[D], dq[D];
    load_row<D>(a.Z + row, z);
    store_row<D>(a.dZ + row, x);
    a.c_out[(size_t)bh * a.M + m] = dot<D>(x, z);
    sum_splits<D>(a.part2, bh, a.tiles, a.splits, m, dq);
    store_row<D>(a.dQ + row, dq);
  } else if (kMode == kLatEnc) {
    float dq[D], qd[D], f[D];
    load_row<D>(a.dQ + row, dq);
#pragma unroll
    for (int d = 0; d < D; ++d) dq[d] += x[d];
    load_row<D>(a.Qd + row, qd);
    const float g = a.gate[h];
    a.dg_part[(size_t)bh * a.M + m] = dot<D>(dq, qd);
    // gate (eq. 7): dQd = g dQ, and c of the synthesis = <dQd, Qd>
    float dqd[D];
#pragma unroll
    for (int d = 0; d < D; ++d) dqd[d] = g * dq[d];
    store_row<D>(a.dQd + row, dqd);
    a.c_out[(size_t)bh * a.M + m] = dot<D>(dqd, qd);
    // N0 of the fixed queries: dQf = r (dQ - y <dQ, y> / D), y = N0(Qf)
    load_t<T, D>(static_cast<const T*>(a.Qf) + ((size_t)h * a.M + m) * D, f);
    const float r = rsqrtf(dot<D>(f, f) / (float)D + kEps);
#pragma unroll
    for (int d = 0; d < D; ++d) f[d] *= r;
    const float proj = dot<D>(dq, f) / (float)D;
#pragma unroll
    for (int d = 0; d < D; ++d) f[d] = r * (dq[d] - f[d] * proj);
    store_row<D>(a.dqf_part + row, f);
  } else {
    store_row<D>(a.dqs_part + row, x);
  }
}

// The per-head parameters' gradients: sums over the batch in a fixed order.
__global__ void reduce_params_kernel(int B, int H, int M, int D, const float* dqs_part, const float* dqf_part,
                                     const float* dg_part, float* dQseed, float* dQf, float* dgate) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int per_head = M * D;
  if (i < H * per_head) {
    const int h = i / per_head, e = i % per_head;
    float a = 0.f, b = 0.f;
    for (int bb = 0; bb < B; ++bb) {
      const size_t off = (size_t)(bb * H + h) * per_head + e;
      a += dqs_part[off];
      b += dqf_part[off];
    }
    dQseed[i] = a;
    dQf[i] = b;
  }
  if (i < H) {
    float g = 0.f;
    for (int bb = 0; bb < B; ++bb)
      for (int m = 0; m < M; ++m) g += dg_part[(size_t)(bb * H + i) * M + m];
    dgate[i] = g;
  }
}

}  // namespace bwd

// ------------------------------------------------------------------ host
namespace {

using namespace bwd;

struct BwdPlan {
  int BH, tiles, splits, split_len;
  size_t off_pz, off_pl, off_cnt, off_qt, off_zt, off_q, off_qd, off_z, off_lenc, off_lsyn, off_ldec,
      off_cdec, off_part2, off_dz, off_dq, off_dqd, off_cenc, off_csyn, off_dqs, off_dqf, off_dg, total;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

BwdPlan make_bwd_plan(int B, int H, int N, int M, int D, bool bf16, int sms) {
  BwdPlan pl{};
  pl.BH = B * H;
  pl.tiles = (M + kRows - 1) / kRows;
  const int max_splits = std::max(1, (N + kTileTok - 1) / kTileTok);
  const long long groups = (long long)pl.BH * pl.tiles;
  const long long want = std::max<long long>(1, (2LL * std::max(sms, 1) + groups - 1) / groups);
  const int splits = (int)std::min<long long>(std::min<long long>(want, 256), max_splits);
  int split_len = (N + splits - 1) / splits;
  split_len = (split_len + kTileTok - 1) / kTileTok * kTileTok;
  pl.split_len = split_len;
  pl.splits = (N + split_len - 1) / split_len;
  const size_t rows = (size_t)pl.BH * pl.tiles * pl.splits * kRows;
  const size_t lat = (size_t)pl.BH * M * D;
  const size_t es = bf16 ? 2 : 4;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = up256(off + bytes); return o; };
  pl.off_pz = take(rows * D * 4);  // forward partials; later the first backward partials
  pl.off_pl = take(rows * 4);
  pl.off_cnt = take(2 * (size_t)pl.BH * pl.tiles * 4);
  pl.off_qt = take(lat * es);
  pl.off_zt = take(lat * es);
  pl.off_q = take(lat * 4);
  pl.off_qd = take(lat * 4);
  pl.off_z = take(lat * 4);
  pl.off_lenc = take((size_t)pl.BH * M * 4);
  pl.off_lsyn = take((size_t)pl.BH * M * 4);
  pl.off_ldec = take((size_t)pl.BH * N * 4);
  pl.off_cdec = take((size_t)pl.BH * N * 4);
  pl.off_part2 = take(rows * D * 4);
  pl.off_dz = take(lat * 4);
  pl.off_dq = take(lat * 4);
  pl.off_dqd = take(lat * 4);
  pl.off_cenc = take((size_t)pl.BH * M * 4);
  pl.off_csyn = take((size_t)pl.BH * M * 4);
  pl.off_dqs = take(lat * 4);
  pl.off_dqf = take(lat * 4);
  pl.off_dg = take((size_t)pl.BH * M * 4);
  pl.total = off;
  return pl;
}

template <typename T, int D>
cudaError_t run_typed(const BwdProblem& p, const BwdPlan& pl, char* ws, cudaStream_t stream, const char** failed) {
  auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  const int BH = pl.BH, M = p.M, N = p.N;
  cudaError_t e;
  *failed = "cudaMemsetAsync(counters)";
  if ((e = cudaMemsetAsync(ws + pl.off_cnt, 0, 2 * (size_t)BH * pl.tiles * 4, stream)) != cudaSuccess) return e;
  // ---- recompute the synthesis and the encode, keeping what the backward reads
  const dim3 grid(pl.splits, pl.tiles, BH);
  simt::SplitArgs<T> sa{};
  sa.H = p.H; sa.N = N; sa.M = M;
  sa.tiles = pl.tiles; sa.splits = pl.splits; sa.split_len = pl.split_len;
  sa.part.z = F(pl.off_pz);
  sa.part.l = F(pl.off_pl);
  sa.part.counters = reinterpret_cast<unsigned*>(ws + pl.off_cnt);
  sa.keys = static_cast<const T*>(p.Ks);
  sa.values = static_cast<const T*>(p.Ks);
  sa.queries = static_cast<const T*>(p.Qseed);
  sa.q_by_head = 1;
  sa.qf = static_cast<const T*>(p.Qf);
  sa.gate = p.gate;
  sa.out = reinterpret_cast<T*>(ws + pl.off_qt);
  sa.dbg_a = F(pl.off_qd);
  sa.dbg_b = F(pl.off_q);
  sa.dbg_c = F(pl.off_lsyn);
  simt::split_kernel<T, D, kPassSynthShared><<<grid, simt::kRows, 0, stream>>>(sa);
  *failed = "launch synthesis (recompute)";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  simt::SplitArgs<T> ea = sa;
  ea.keys = static_cast<const T*>(p.K);
  ea.values = static_cast<const T*>(p.V);
  ea.queries = reinterpret_cast<const T*>(ws + pl.off_qt);
  ea.q_by_head = 0;
  ea.qf = nullptr;
  ea.gate = nullptr;
  ea.part.counters = reinterpret_cast<unsigned*>(ws + pl.off_cnt) + (size_t)BH * pl.tiles;
  ea.out = reinterpret_cast<T*>(ws + pl.off_zt);
  ea.dbg_a = F(pl.off_z);
  ea.dbg_b = F(pl.off_lenc);
  ea.dbg_c = nullptr;
  simt::split_kernel<T, D, kPassEncode><<<grid, simt::kRows, 0, stream>>>(ea);
  *failed = "launch encode (recompute)";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const dim3 tgrid((N + kRows - 1) / kRows, BH);
  const size_t smem2 = 2 * (size_t)M * D * 4, smem2l = smem2 + 2 * (size_t)M * 4;
  const int mgrid = (BH * M + 127) / 128;
  // ---- decode: token-major, then latent-major and its merge
  *failed = "cudaFuncSetAttribute(backward)";
  if ((e = cudaFuncSetAttribute(dec_token_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2)) ||
      (e = cudaFuncSetAttribute(enc_token_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2l)) ||
      (e = cudaFuncSetAttribute(syn_token_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2l)))
    return e;
  dec_token_kernel<T, D><<<tgrid, kRows, smem2, stream>>>(static_cast<const T*>(p.K), static_cast<const T*>(p.dY),
                                                          F(pl.off_q), F(pl.off_z), N, M, p.dK, F(pl.off_ldec),
                                                          F(pl.off_cdec));
  *failed = "launch dec_token_kernel";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  LatArgs<T> la{};
  la.H = p.H; la.N = N; la.M = M;
  la.tiles = pl.tiles; la.splits = pl.splits; la.split_len = pl.split_len;
  la.part1 = F(pl.off_pz);
  la.part2 = F(pl.off_part2);
  la.keys = static_cast<const T*>(p.K);
  la.vals = static_cast<const T*>(p.dY);
  la.tok_l = F(pl.off_ldec);
  la.tok_c = F(pl.off_cdec);
  la.lat_q = F(pl.off_q);
  la.lat_o = F(pl.off_z);
  latent_kernel<T, D, kLatDec><<<grid, kRows, 0, stream>>>(la);
  *failed = "launch latent_kernel (decode)";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  MergeArgs ma{};
  ma.H = p.H; ma.M = M; ma.tiles = pl.tiles; ma.splits = pl.splits;
  ma.part1 = F(pl.off_pz);
  ma.part2 = F(pl.off_part2);
  ma.Z = F(pl.off_z);
  ma.Qd = F(pl.off_qd);
  ma.Qf = p.Qf;
  ma.gate = p.gate;
  ma.dZ = F(pl.off_dz);
  ma.dQ = F(pl.off_dq);
  ma.c_out = F(pl.off_cenc);
  ma.dQd = F(pl.off_dqd);
  ma.dg_part = F(pl.off_dg);
  ma.dqf_part = F(pl.off_dqf);
  ma.dqs_part = F(pl.off_dqs);
  merge_kernel<T, D, kLatDec><<<mgrid, 128, 0, stream>>>(ma, BH);
  *failed = "launch merge_kernel (decode)";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // ---- encode
  enc_token_kernel<T, D><<<tgrid, kRows, smem2l, stream>>>(static_cast<const T*>(p.K), static_cast<const T*>(p.V),
                                                           F(pl.off_q), F(pl.off_dz), F(pl.off_lenc),
                                                           F(pl.off_cenc), N, M, p.dK, p.dV);
  *failed = "launch enc_token_kernel";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  LatArgs<T> le = la;
  le.vals = static_cast<const T*>(p.V);
  le.tok_l = nullptr;
  le.tok_c = nullptr;
  le.lat_o = F(pl.off_dz);
  le.lat_l = F(pl.off_lenc);
  le.lat_c = F(pl.off_cenc);
  le.part2 = nullptr;
  latent_kernel<T, D, kLatEnc><<<grid, kRows, 0, stream>>>(le);
  *failed = "launch latent_kernel (encode)";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  MergeArgs me = ma;
  me.c_out = F(pl.off_csyn);
  merge_kernel<T, D, kLatEnc><<<mgrid, 128, 0, stream>>>(me, BH);
  *failed = "launch merge_kernel (encode)";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // ---- synthesis
  syn_token_kernel<T, D><<<tgrid, kRows, smem2l, stream>>>(static_cast<const T*>(p.Ks),
                                                           static_cast<const T*>(p.Qseed), F(pl.off_dqd),
                                                           F(pl.off_lsyn), F(pl.off_csyn), N, M, p.H, p.dKs);
  *failed = "launch syn_token_kernel";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  LatArgs<T> ls = la;
  ls.keys = static_cast<const T*>(p.Ks);
  ls.vals = nullptr;
  ls.tok_l = nullptr;
  ls.tok_c = nullptr;
  ls.lat_q = nullptr;
  ls.seeds = static_cast<const T*>(p.Qseed);
  ls.lat_o = F(pl.off_dqd);
  ls.lat_l = F(pl.off_lsyn);
  ls.lat_c = F(pl.off_csyn);
  ls.part2 = nullptr;
  latent_kernel<T, D, kLatSyn><<<grid, kRows, 0, stream>>>(ls);
  *failed = "launch latent_kernel (synthesis)";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  merge_kernel<T, D, kLatSyn><<<mgrid, 128, 0, stream>>>(ma, BH);
  *failed = "launch merge_kernel (synthesis)";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int rn = std::max(p.H * M * D, p.H);
  reduce_params_kernel<<<(rn + 255) / 256, 256, 0, stream>>>(p.B, p.H, M, D, F(pl.off_dqs), F(pl.off_dqf),
                                                             F(pl.off_dg), p.dQseed, p.dQf, p.dgate);
  *failed = "launch reduce_params_kernel";
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  *failed = "";
  return cudaSuccess;
}

}  // namespace

size_t backward_workspace_bytes(int B, int H, int N, int M, int D, bool bf16, int sms) {
  return make_bwd_plan(B, H, N, M, D, bf16, sms).total;
}

cudaError_t backward_run(const BwdProblem& p, void* ws, size_t ws_bytes, int sms, cudaStream_t stream,
                         const char** failed) {
  const BwdPlan pl = make_bwd_plan(p.B, p.H, p.N, p.M, p.D, p.bf16, sms);
  *failed = "backward workspace too small";
  if (ws_bytes < pl.total) return cudaErrorInvalidValue;
  char* w = static_cast<char*>(ws);
  if (p.bf16)
    return p.D == 16 ? run_typed<__nv_bfloat16, 16>(p, pl, w, stream, failed)
                     : run_typed<__nv_bfloat16, 32>(p, pl, w, stream, failed);
  return p.D == 16 ? run_typed<float, 16>(p, pl, w, stream, failed)
                   : run_typed<float, 32>(p, pl, w, stream, failed);
}

}  // namespace flarepp
