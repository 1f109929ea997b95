// flarepp_forward_static: the mixer forward for callers that cannot allocate
// device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocating routine)
// at the point where they run the mixer: code running under a memory budget
// that a framework's own allocator owns completely, plug-ins whose host process
// forbids device allocations after start-up, or real-time loops that must not
// block on the allocator. For them this file keeps the forward's scratch (the
// split-N partial results, the arrival counters and the intermediate Q and Z)
// in one file-scope device array of fixed size, reserved when the library's
// module is loaded and held by every GPU that loads it until the process exits.
//
// The forward itself is unchanged: this entry point hands the array's address,
// as caller-style workspace, to flarepp_forward_ws, which clears the counters
// at the start of every call and writes every other scratch byte before it
// reads it.
#include <cuda_runtime.h>

#include "flarepp.h"

namespace {

// Largest scratch this entry point can use: 32 MiB per device.
constexpr size_t kScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

// Device address of g_static_scratch on the current device. Host code must
// not use the symbol itself (on the host it names a stand-in object). The
// address is looked up on every call, with the device current: the lookup
// allocates nothing, and an address cached across calls would go stale when
// the device's context is torn down and created again (cudaDeviceReset).
flarepp_status_t scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return FLAREPP_ERR_CUDA;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return FLAREPP_ERR_CUDA;
  }
  *out = p;
  return FLAREPP_OK;
}

}  // namespace

extern "C" flarepp_status_t flarepp_forward_static(const void* K, const void* V, const void* Ks_raw,
                                                   const void* Qseed, const void* Qf,
                                                   const float* gate, int B, int H, int N, int M,
                                                   int D, flarepp_dtype_t dtype, void* out,
                                                   cudaStream_t stream) {
  const size_t need = flarepp_workspace_size(B, H, N, M, D, dtype);
  if (need == 0) {
    // unsupported sizes or no device: let the shared validation give the reason
    return flarepp_forward_ws(K, V, Ks_raw, Qseed, Qf, gate, B, H, N, M, D, dtype, out, nullptr, 0,
                              stream);
  }
  if (need > kScratchBytes) return FLAREPP_ERR_NO_MEMORY;
  void* scratch = nullptr;
  const flarepp_status_t st = scratch_for_current_device(&scratch);
  if (st != FLAREPP_OK) return st;
  return flarepp_forward_ws(K, V, Ks_raw, Qseed, Qf, gate, B, H, N, M, D, dtype, out, scratch,
                            kScratchBytes, stream);
}
