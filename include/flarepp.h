/*
 * flarepp.h — C ABI of the GB300 (sm_103a) FLARE++ mixer forward.
 *
 * The operation is the token mixer of "FLARE++: Low-rank attention with
 * attention-synthesized routing" (arXiv 2608.11519 v2), Section 3.2, for each
 * batch entry b and head h independently, with s = 1/sqrt(D):
 *
 *   Kt  = N0(Ks_raw)                          eq. 5  (RMSNorm, no scale, eps 1e-6)
 *   Qd  = softmax_N(s Qseed Kt^T) Kt          eq. 6 / eq. 19 (keys shared as values)
 *   Q   = N0(Qf) + g Qd   (fp32, then cast)   eq. 7 / eq. 15
 *   Z   = softmax_N(s Q K^T) V,  L = LSE_N    eq. 8, Appendix B.2 eq. 23-25
 *   out = softmax_M(s K Q^T) Z                eq. 8 (decode softmax over the M routes)
 *
 * Conventions for every entry point below:
 *   - All tensor pointers are DEVICE pointers on the device that `stream`
 *     belongs to, contiguous and row-major, 16-byte aligned.
 *   - K, V, Ks_raw, out: [B, H, N, D] of `dtype`.  Qseed, Qf: [H, M, D] of
 *     `dtype`.  gate: [H] fp32, the post-sigmoid value g in [0, 1).
 *   - K is the routing key as used (the caller applies its learned-scale
 *     RMSNorm N_a); Qseed is the seed as used (N_a already applied); Ks_raw is
 *     taken before N0, and Qf before N0 — the library applies both N0s.
 *   - N is the exact token count of every batch entry; there is no mask.
 *   - Supported: D in {16, 32}; 1 <= M <= 512 (bf16: M % 16 == 0); N >= 1;
 *     B*H*N*D < 2^31 elements per tensor.
 *   - The caller owns every buffer. The library keeps no pointer after return.
 *   - Calls are asynchronous on `stream`; a returned FLAREPP_OK means the work
 *     was enqueued. Argument errors are detected before anything is launched.
 *   - No C++ exception crosses this interface.
 */
#ifndef FLAREPP_H_
#define FLAREPP_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FLAREPP_BF16 = 0, FLAREPP_FP32 = 1 } flarepp_dtype_t;

typedef enum {
  FLAREPP_OK = 0,
  FLAREPP_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, out aliasing an input */
  FLAREPP_ERR_UNSUPPORTED = 2,  /* D, M or dtype outside the supported set */
  FLAREPP_ERR_ALIGNMENT = 3,    /* a pointer not 16-byte aligned */
  FLAREPP_ERR_NO_MEMORY = 4,    /* workspace could not be allocated or is too small */
  FLAREPP_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed */
  FLAREPP_ERR_TIMEOUT = 6       /* a device-side bounded wait gave up (see flarepp_sync_status) */
} flarepp_status_t;

/*
 * The full mixer forward (all six steps above) for B batch entries and H
 * heads, writing out[B,H,N,D]. Workspace comes from a per-device,
 * per-stream cache inside the library (stream-ordered cudaMallocAsync,
 * guarded by a mutex); it grows on demand and is reused across calls on the
 * same stream. Use flarepp_forward_ws to pass workspace explicitly instead.
 */
flarepp_status_t flarepp_forward(const void* K, const void* V, const void* Ks_raw,
                                 const void* Qseed, const void* Qf, const float* gate,
                                 int B, int H, int N, int M, int D, flarepp_dtype_t dtype,
                                 void* out, cudaStream_t stream);

/*
 * Bytes of device workspace that flarepp_forward_ws needs for these sizes
 * (split-N partial results, arrival counters, the routing queries Q and the
 * latents Z). Returns 0 if the sizes are unsupported.
 */
size_t flarepp_workspace_size(int B, int H, int N, int M, int D, flarepp_dtype_t dtype);

/*
 * As flarepp_forward, with caller-owned device workspace of at least
 * flarepp_workspace_size(...) bytes, 256-byte aligned. The library allocates
 * nothing on this path. Two calls that run at the same time on the GPU must
 * not share one workspace.
 */
flarepp_status_t flarepp_forward_ws(const void* K, const void* V, const void* Ks_raw,
                                    const void* Qseed, const void* Qf, const float* gate,
                                    int B, int H, int N, int M, int D, flarepp_dtype_t dtype,
                                    void* out, void* workspace, size_t ws_bytes,
                                    cudaStream_t stream);

/*
 * As flarepp_forward, and also copies the intermediate results of the
 * steps, each as fp32 device arrays (any may be NULL):
 *   Qd_out [B,H,M,D] the merged synthesis output of eq. 6 (before the gate);
 *   Q_out  [B,H,M,D] the routing queries of eq. 7 as the kernels use them
 *                    (rounded to `dtype`);
 *   Z_out  [B,H,M,D] the encoded latents of eq. 8 as used by the decode
 *                    (rounded to `dtype`);
 *   L_out  [B,H,M]   the encode log-normaliser (natural log).
 */
flarepp_status_t flarepp_forward_debug(const void* K, const void* V, const void* Ks_raw,
                                       const void* Qseed, const void* Qf, const float* gate,
                                       int B, int H, int N, int M, int D, flarepp_dtype_t dtype,
                                       void* out, float* Qd_out, float* Q_out, float* Z_out,
                                       float* L_out, cudaStream_t stream);

/*
 * As flarepp_forward_ws, for callers that cannot allocate device memory: the
 * scratch lives in one fixed array inside the library (32 MiB per device,
 * reserved when the library's device code is loaded and kept until the process
 * exits), so the call itself allocates nothing. The FLARE++ paper has no
 * counterpart; this exists for host programs whose allocator owns all device
 * memory, or that may not allocate after start-up, or that must not block on
 * an allocation inside a timed loop.
 *   - Returns FLAREPP_ERR_NO_MEMORY when these sizes need more scratch than
 *     the 32 MiB maximum (flarepp_workspace_size(...) > 32 MiB).
 *   - Every call looks up the array's device address with the device current
 *     (a lookup, no allocation). The first call on a device may also load the
 *     library's device code there; make that first call before any stream
 *     capture.
 *   - All calls on a device share the one array, and it keeps the previous
 *     call's contents (the library clears what must start at zero). Calls that
 *     overlap on the GPU — on different streams, or from different host threads
 *     without ordering between them — race on it and give wrong results;
 *     serialise them.
 */
flarepp_status_t flarepp_forward_static(const void* K, const void* V, const void* Ks_raw,
                                        const void* Qseed, const void* Qf, const float* gate,
                                        int B, int H, int N, int M, int D, flarepp_dtype_t dtype,
                                        void* out, cudaStream_t stream);

/*
 * The two synthesis variants that the FLARE++ paper defines beside the
 * default mixer above (Appendix A.1 and A.8), for flarepp_forward_variant.
 */
typedef enum {
  /* The default mixer above: Vs must be NULL (eq. 5-8, eq. 19). */
  FLAREPP_VARIANT_SHARED = 0,
  /* The general form with a separate synthesis value projection (Appendix
   * A.1, eq. 11):  Qd = softmax_N(s Qseed N0(Ks_raw)^T) Vs, then
   * Q = N0(Qf) + g Qd and eq. 8 as above. Vs [B,H,N,D] is used as given (the
   * library normalises only the synthesis keys); Vs = N0(Ks_raw) gives the
   * default mixer. */
  FLAREPP_VARIANT_UNSHARED = 1,
  /* Simplified FLARE++ (Appendix A.8, eq. 20):  Q = Qd =
   * softmax_N(s Qseed Ks^T) Vs, rounded to `dtype`, then eq. 8. No fixed
   * reference and no gate: Qf and gate must be NULL. Qseed and Ks are taken
   * as used (the caller applies their learned-scale RMSNorms N_a; the library
   * applies no N0 here); Vs is the unnormalised value projection. */
  FLAREPP_VARIANT_SIMPLIFIED = 2
} flarepp_variant_t;

/*
 * The mixer forward for one of the variants above. Arguments as for
 * flarepp_forward, plus:
 *   Ks     [B,H,N,D] the synthesis keys (Ks_raw of flarepp_forward for SHARED
 *          and UNSHARED, which apply N0; used as given by SIMPLIFIED);
 *   Vs     [B,H,N,D] the separate synthesis values (UNSHARED, SIMPLIFIED;
 *          NULL for SHARED).
 *   Qf, gate: required by SHARED and UNSHARED, NULL for SIMPLIFIED.
 * Optional fp32 copies of the intermediate results as in
 * flarepp_forward_debug (each may be NULL); SIMPLIFIED has no separate Qd
 * (Q is Qd) and leaves Qd_out untouched. A pointer that the variant does not
 * read but is not NULL, or one it reads that is NULL, gives
 * FLAREPP_ERR_INVALID_ARG. Workspace comes from the per-stream cache, as for
 * flarepp_forward. Supported sizes and dtypes as for flarepp_forward.
 */
flarepp_status_t flarepp_forward_variant(flarepp_variant_t variant, const void* K, const void* V,
                                         const void* Ks, const void* Vs, const void* Qseed,
                                         const void* Qf, const float* gate, int B, int H, int N,
                                         int M, int D, flarepp_dtype_t dtype, void* out,
                                         float* Qd_out, float* Q_out, float* Z_out, float* L_out,
                                         cudaStream_t stream);

/*
 * FLARE, the fixed-query latent routing that FLARE++ builds on (Section 3.1,
 * eq. 2-3): each head h routes through its own learned query set Q_h,
 *   Z = softmax_N(s Q_h K^T) V,   out = softmax_M(s K Q_h^T) Z,
 * the encode and decode steps of flarepp_forward without the synthesis.
 *   Q      [H,M,D] of `dtype`, used as given (no normalisation);
 *   K, V, out [B,H,N,D] as for flarepp_forward;
 *   Z_out  [B,H,M,D] optional fp32 copy of the latents as the decode reads
 *          them (rounded to `dtype`); L_out [B,H,M] optional fp32 encode
 *          log-normaliser (natural log); either may be NULL.
 * Sizes, dtypes, alignment, ownership, asynchrony and errors as for
 * flarepp_forward; workspace from the same per-stream cache.
 */
flarepp_status_t flare_forward(const void* Q, const void* K, const void* V, int B, int H, int N, int M,
                               int D, flarepp_dtype_t dtype, void* out, float* Z_out, float* L_out,
                               cudaStream_t stream);

/* Per-head normalisation of a projection's output (flarepp_project). */
typedef enum {
  FLAREPP_NORM_NONE = 0, /* none */
  FLAREPP_NORM_N0 = 1,   /* RMSNorm over D without scale, eps 1e-6 (N0 of Section 3.2) */
  FLAREPP_NORM_NA = 2    /* RMSNorm over D with a learned scale of D values (N_a) */
} flarepp_norm_t;

/*
 * The pointwise token projections that produce the mixer's inputs
 * (Section 3.2 and Appendix A.7 Table 2 of the paper: K = N_a(X W_K),
 * V = X W_V, the synthesis keys X W~_K; or the simplified variant's set),
 * P of them in one pass over X:
 *
 *   outs[p][b, h, n, d] = norm_p( X[b, n, :] . W[p*C + h*D + d, :] + bias[p*C + h*D + d] )
 *
 * with C = H*D, the norm applied to each head's D values (bias first).
 *   X      [B, N, C] of `dtype` (device), the block input after its pre-norm;
 *   W      [P*C, C] of `dtype` (device): the P weight matrices stacked, each in
 *          the out x in layout of a linear layer, output channel h*D + d
 *          belonging to head h;
 *   bias   [P*C] fp32 (device) or NULL;
 *   norms  P codes (HOST array);
 *   scales [P, D] fp32 (device): row p is the N_a scale of output p; NULL
 *          exactly when no output uses FLAREPP_NORM_NA;
 *   outs   P DEVICE pointers (HOST array), each [B, H, N, D] of `dtype`, the
 *          layout flarepp_forward takes. They must not overlap each other or
 *          any input.
 * Supported: 1 <= P <= 4; D in {16, 32}; bf16 needs C in {64, 128, 256},
 * fp32 C <= 256; B <= 65535; B*H*N*D < 2^31. The bf16 path rounds each output
 * once (fp32 accumulation, bias and norm in fp32). Alignment, ownership,
 * asynchrony and errors as for flarepp_forward; the call needs no workspace.
 */
flarepp_status_t flarepp_project(const void* X, const void* W, const float* bias, int P,
                                 const flarepp_norm_t* norms, const float* scales, void* const* outs,
                                 int B, int H, int N, int D, flarepp_dtype_t dtype,
                                 cudaStream_t stream);

/*
 * Backward pass of the mixer (flarepp_forward): given the cotangent dY of the
 * output, the gradients of every input,
 *   dK, dV, dKs_raw [B,H,N,D], dQseed, dQf [H,M,D] (summed over the batch),
 *   dgate [H] (summed over the batch and the routes),
 * all fp32 DEVICE arrays whatever `dtype` is. The inputs are those of
 * flarepp_forward plus dY [B,H,N,D] of `dtype`. Each attention call is
 * differentiated with the local backward of Appendix B.5 (eq. 46-49: the
 * merged log-normaliser recovers the probabilities, c = <dOut, Out> per row,
 * no cotangent on L); the gate (eq. 7) and both N0s follow by the chain rule.
 * The call recomputes the forward's synthesis and encode (nothing has to be
 * kept from the forward) and runs in fp32 arithmetic on the CUDA cores; for
 * bf16 it uses Q and Z rounded to bf16, as the forward does. Results are
 * bitwise repeatable (every reduction has a fixed order). Workspace comes
 * from the per-stream cache of flarepp_forward. Sizes, alignment, ownership,
 * asynchrony and errors as for flarepp_forward; the outputs must not overlap
 * each other or any input.
 */
flarepp_status_t flarepp_backward(const void* K, const void* V, const void* Ks_raw, const void* Qseed,
                                  const void* Qf, const float* gate, const void* dY, int B, int H, int N,
                                  int M, int D, flarepp_dtype_t dtype, float* dK, float* dV, float* dKs_raw,
                                  float* dQseed, float* dQf, float* dgate, cudaStream_t stream);

/*
 * Waits for `stream`, then reports (and clears) any device-side error that
 * the library's kernels recorded since the last call on this device:
 * FLAREPP_ERR_TIMEOUT if a bounded wait gave up, FLAREPP_ERR_CUDA if the
 * stream reported a CUDA error, FLAREPP_OK otherwise.
 */
flarepp_status_t flarepp_sync_status(cudaStream_t stream);

/* A static, human-readable name of a status code. Never NULL. */
const char* flarepp_status_string(flarepp_status_t status);

/*
 * Which CUDA call last failed on the calling thread, with CUDA's error name
 * and text ("no error" if none). The string is owned by the library and valid
 * until the thread's next library call.
 */
const char* flarepp_last_error(void);

/*
 * Test hook: the number of token splits per (batch, head) that the next calls
 * use for the two split-N passes; 0 restores the automatic choice. The result
 * does not depend on the split count beyond floating-point rounding (the
 * log-sum-exp merge of Appendix B.2-B.3 is exact in exact arithmetic).
 */
void flarepp_set_splits(int splits);

/*
 * Pipeline trace, for builds compiled with FLAREPP_TRACE (otherwise
 * FLAREPP_ERR_UNSUPPORTED). pass 1 (synthesis), 2 (encode) or 3 (decode)
 * arms the trace: block 0 of that pass records clock64 stamps of its
 * pipeline events in the next calls; 0 disarms. When `host` is not NULL,
 * up to n stamps (16 roles x 4096 events, role-major) are copied to it.
 * Synchronous; not thread-safe: for profiling.
 */
flarepp_status_t flarepp_debug_trace(int pass, unsigned long long* host, int n);

/*
 * Test hook for the device-side failure path (the FLARE++ paper has no
 * counterpart): while `pass` is 1 (synthesis), 2 (encode) or 3 (decode), the
 * bf16 forward calls make one barrier of that pass expect an arrival that
 * never comes, and every bounded wait of that pass gives up after about a
 * millisecond instead of a second. The MMA-issuing thread waiting on the
 * barrier gives up, records the timeout and makes its CTA leave;
 * the call's output is then undefined and flarepp_sync_status returns
 * FLAREPP_ERR_TIMEOUT. 0 (or any other value) switches it off. No fault,
 * trap or unbounded wait is involved, and the context stays usable. Not
 * thread-safe: for tests.
 */
void flarepp_test_fail_wait(int pass);

/*
 * Measurement hook: while set (events != NULL, count >= 4), every forward call
 * records events[0] before its first kernel, events[1] after the synthesis
 * pass (steps a1-a3), events[2] after the encode pass (a4-a5) and events[3]
 * after the decode (a6), all on the call's stream, so cudaEventElapsedTime
 * gives each pass's device time. The array is caller-owned and must outlive
 * the calls; pass NULL to clear. Not thread-safe: for benchmarks and tests.
 */
void flarepp_set_stage_events(cudaEvent_t* events, int count);

/*
 * Planning hook: the launch plan that flarepp_forward would use for these
 * sizes on a GPU with `sms` multiprocessors, computed on the host without
 * touching a device (for tests and tuning; the FLARE++ paper has no
 * counterpart). Writes min(n, 8) values to `fields`:
 *   [0] token splits per (batch, head, latent group) of the synthesis and
 *       encode passes (respects flarepp_set_splits);
 *   [1] tokens per split (a multiple of the 128-token tile on the bf16 path);
 *   [2] latent groups per (batch, head): CTAs that split the M latent rows;
 *   [3] consecutive 128-token tiles per decode CTA;
 *   [4] decode CTAs per (batch, head), or 0 when the decode CTAs walk the
 *       flattened (batch, head, tile) order and may span heads;
 *   [5] heads whose Q and Z one decode CTA keeps in shared memory;
 *   [6] decode CTAs in all;
 *   [7] workspace bytes (as flarepp_workspace_size), clamped to INT_MAX.
 * Fields [2]-[6] are 0 on the fp32 path, whose kernels plan differently.
 * Returns FLAREPP_OK, FLAREPP_ERR_INVALID_ARG (fields NULL, n < 1 or
 * sms < 1) or the size check's status (FLAREPP_ERR_UNSUPPORTED, ...).
 */
flarepp_status_t flarepp_plan_info(int B, int H, int N, int M, int D, flarepp_dtype_t dtype,
                                   int sms, int* fields, int n);

#ifdef __cplusplus
}
#endif

#endif /* FLAREPP_H_ */
