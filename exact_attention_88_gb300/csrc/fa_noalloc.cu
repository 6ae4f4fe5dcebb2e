// fa_bwd_noalloc: the bf16 backward pass for callers that cannot allocate
// device memory.
//
// fa_bwd needs a workspace (the per-row D vector) that the caller allocates.  Some callers cannot do that: a plugin running
// inside a host framework that has already reserved all device memory for its
// own pool and forbids extensions from calling cudaMalloc, or latency-critical
// code that must not call cudaMalloc/cudaFree because they can synchronize
// the whole device.  This entry point takes its workspace from a fixed array
// compiled into the library instead.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes; every
// GPU that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address (on the host it names a
// host-side stand-in), so the first call on each device looks up its device
// address with cudaGetSymbolAddress, with that device current, and caches it.
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = FA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxNoAllocDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device, looked up once
// per device.  On failure returns the CUDA error and leaves *out unset.
cudaError_t scratch_address(void** out) {
  static void* addr[kMaxNoAllocDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxNoAllocDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    const void* dO, const float* lse, void* dq, void* dk,
                                    void* dv, int B, int H, int N, int d, float scale, int causal,
                                    const fa_mask* mask, void* stream) {
  // fa_bwd's own argument checks first, on the host only, so that argument
  // errors come back with fa_bwd's codes before any CUDA runtime call
  fa_status st = fa::check_bwd_args(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal,
                                    mask);
  if (st != FA_OK) return st;
  if (fa_bwd_workspace_size(B, H, N, d) > fa::kNoAllocScratchBytes)
    return FA_ERR_UNSUPPORTED;  // beyond the fixed scratch
  void* scratch = nullptr;
  st = fa::cuda_status(fa::scratch_address(&scratch));
  if (st != FA_OK) return st;
  // fa_bwd writes D into the scratch before any kernel reads it, then runs
  // the backward kernels on `stream`.
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, scratch, fa::kNoAllocScratchBytes, B, H, N, d,
                scale, causal, mask, stream);
}
