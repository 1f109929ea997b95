// Interface between the host API (flarepp.cu) and the tensor-core kernels
// (tc.cu): one problem description and the launch entry of each kernel family.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace flarepp {

// Which mixer of the FLARE++ paper a call computes.
enum Variant : int {
  kVariantFlarePP = 0,     // eq. 5-8, synthesis keys shared as values (eq. 19)
  kVariantUnshared = 1,    // eq. 11: separate synthesis values Vs
  kVariantSimplified = 2,  // eq. 20: Q = SDPA(Qseed, Ks, Vs); no reference, no gate
  kVariantFlare = 3,       // eq. 3: the caller's learned queries Q, no synthesis
};

// One forward call as the kernels see it. All pointers are device pointers;
// those a variant does not use are null.
struct DeviceProblem {
  int variant;         // Variant
  const void* K;       // [BH][N][D]
  const void* V;       // [BH][N][D]
  const void* Ks;      // [BH][N][D] synthesis keys (raw for the N0 variants)
  const void* Vs;      // [BH][N][D] separate synthesis values
  const void* Qseed;   // [H][M][D]
  const void* Qf;      // [H][M][D]
  const float* gate;   // [H]
  const void* Q;       // [H][M][D] FLARE's learned queries
  void* out;           // [BH][N][D]
  int B, H, N, M, D;
  float* dbg_qd;       // optional fp32 copies of the intermediate results
  float* dbg_q;
  float* dbg_z;
  float* dbg_l;
  int fail_wait;       // test only: pass (1 synthesis, 2 encode, 3 decode) whose first P barrier never completes
};

// Split-N layout shared by the synthesis and encode passes: `tiles` blocks of
// (up to) 128 latent rows per head, handled by `qgroups` CTAs per token split
// (one block per CTA); `splits` token ranges of `split_len`
// tokens (a multiple of 128); `streams` partial results per (block, split,
// row): 1, the token streams inside a CTA being merged before the write.
struct TcPlan {
  int tiles, qgroups, splits, split_len, streams;
  // decode: tiles per CTA; CTAs per head (0: CTAs walk the flattened
  // (head, tile) order); Q/Z slots per CTA; grid size
  int decode_tiles_per_cta, decode_ctas_per_head, decode_heads, decode_ctas;
};

// Workspace regions (device pointers into the caller's or the cache's buffer).
struct TcWorkspace {
  float* part_z;           // [BH][tiles][splits][128][D]
  float* part_l;           // [BH][tiles][splits][128]
  unsigned* counters;      // [2][BH][tiles]
  void* q;                 // [BH][M][D] bf16 routing queries
  void* z;                 // [BH][M][D] bf16 latents
};

TcPlan tc_plan(int B, int H, int N, int M, int D, int sms, int forced_splits);
// Launches synthesis, encode and decode on `stream`. `events` (4 entries or
// null) bracket the three passes. Returns a cudaError_t of the first failure.
cudaError_t tc_forward(const DeviceProblem& p, const TcPlan& pl, const TcWorkspace& ws,
                       cudaEvent_t* events, cudaStream_t stream, const char** failed_call);
// Reads and clears the tensor-core kernels' device error word (bit 0: a
// bounded wait timed out).
cudaError_t tc_take_error_word(unsigned* word);
cudaError_t tc_trace(int pass, unsigned long long* host, int n);

// ------------------------------------------------------ token projections
constexpr int kMaxProjParts = 4;
enum : int { kNormNone = 0, kNormN0 = 1, kNormNa = 2 };

// Kernel arguments of the projection kernels.
struct ProjParams {
  int N, H, P, tiles, tiles_per_b;
  const float* bias;    // [P*C] or null
  const float* scales;  // [P][D] (rows of N_a parts) or null
  int norms[kMaxProjParts];
};

// One projection call: X [B][N][C] and W [P*C][C] of the model dtype, outputs
// [B][H][N][D] of the same dtype, C = H D. Device pointers.
struct ProjProblem {
  const void* X;
  const void* W;
  const float* bias;
  const float* scales;
  int norms[kMaxProjParts];
  void* outs[kMaxProjParts];
  int P, B, H, N, D;
};

bool proj_supported(int H, int D, bool bf16);
cudaError_t proj_forward(const ProjProblem& p, int sms, bool bf16, cudaStream_t stream, const char** failed_call);
// Reads and clears the projection kernel's device error word.
cudaError_t proj_take_error_word(unsigned* word);

// ------------------------------------------------------------- backward
// One backward call: the forward's inputs and dY of the model dtype, the
// gradients in fp32. Device pointers.
struct BwdProblem {
  const void* K;
  const void* V;
  const void* Ks;
  const void* Qseed;
  const void* Qf;
  const float* gate;
  const void* dY;
  int B, H, N, M, D;
  bool bf16;
  float* dK;      // [B][H][N][D]
  float* dV;      // [B][H][N][D]
  float* dKs;     // [B][H][N][D]
  float* dQseed;  // [H][M][D]
  float* dQf;     // [H][M][D]
  float* dgate;   // [H]
};

size_t backward_workspace_bytes(int B, int H, int N, int M, int D, bool bf16, int sms);
cudaError_t backward_run(const BwdProblem& p, void* ws, size_t ws_bytes, int sms, cudaStream_t stream,
                         const char** failed_call);

}  // namespace flarepp
