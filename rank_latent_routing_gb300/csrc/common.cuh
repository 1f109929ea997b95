// Device helpers shared by the FLARE++ kernels: element loads/stores for the
// two model dtypes, the library's device error word, and the layout of the
// split-N workspace.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace flarepp {

// RMSNorm eps of N0 (FLARE++ paper Section 3.2 eq. 5 gives none; see header).
constexpr float kEps = 1e-6f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device error word: kernels OR bits in here instead of trapping. The whole
// library is one translation unit, so this is its only definition.
enum : unsigned { kErrTimeout = 1u, kErrBadState = 2u };
__device__ unsigned g_error_word = 0u;

__device__ __forceinline__ void record_error(unsigned bits) { atomicOr(&g_error_word, bits); }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Loads `n` (multiple of 4 for fp32, of 8 for bf16) consecutive elements
// starting at a 16-byte aligned address and widens them to fp32.
template <int n>
__device__ __forceinline__ void load_row(const float* p, float* out) {
#pragma unroll
  for (int i = 0; i < n; i += 4) {
    float4 v = __ldg(reinterpret_cast<const float4*>(p + i));
    out[i] = v.x; out[i + 1] = v.y; out[i + 2] = v.z; out[i + 3] = v.w;
  }
}
template <int n>
__device__ __forceinline__ void load_row(const __nv_bfloat16* p, float* out) {
#pragma unroll
  for (int i = 0; i < n; i += 8) {
    uint4 v = __ldg(reinterpret_cast<const uint4*>(p + i));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      out[i + 2 * j] = __uint_as_float(w[j] << 16);
      out[i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

template <int n>
__device__ __forceinline__ void store_row(float* p, const float* v) {
#pragma unroll
  for (int i = 0; i < n; i += 4)
    *reinterpret_cast<float4*>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}
template <int n>
__device__ __forceinline__ void store_row(__nv_bfloat16* p, const float* v) {
#pragma unroll
  for (int i = 0; i < n; i += 8) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[i + 2 * j], v[i + 2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p + i) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Rounds through the model dtype and back (what the next step will read).
template <typename T> __device__ __forceinline__ float round_as(float x) {
  return to_f32(from_f32<T>(x));
}

// What a split-N pass computes (FLARE++ paper):
//  kPassEncode         SDPA(Q, K, V): the encode of eq. 8 and of FLARE's eq. 3,
//                      and the synthesis of the simplified variant (eq. 20);
//  kPassSynthShared    SDPA(Qseed, N0(Ks), N0(Ks)) then the gate (eq. 6-7, 19);
//  kPassSynthSeparate  SDPA(Qseed, N0(Ks), Vs) then the gate (eq. 11).
enum PassKind : int { kPassEncode = 0, kPassSynthShared = 1, kPassSynthSeparate = 2 };

__host__ __device__ constexpr bool pass_normalises_keys(int kind) { return kind != kPassEncode; }
__host__ __device__ constexpr bool pass_separate_values(int kind) { return kind != kPassSynthShared; }
__host__ __device__ constexpr bool pass_gated(int kind) { return kind != kPassEncode; }

// Split-N partial results of one pass (synthesis or encode), per
// (batch*head, row tile of 128 latents, split): Z_s [128][D] fp32 normalised
// by its own split's softmax sum, and L_s [128] its natural-log normaliser
// (FLARE++ Appendix B.2 eq. 25-26 with shards = splits). One arrival counter
// per (batch*head, row tile).
struct Partials {
  float* z;            // [BH][tiles][splits][128][D]
  float* l;            // [BH][tiles][splits][128]
  unsigned* counters;  // [BH][tiles]
};

}  // namespace flarepp
