// The failure-path check: a single-CTA kernel whose only wait can never
// complete, bounded exactly like the attention kernels' waits, so that the
// timeout path (abort flag, status word, host-side FA_ERR_TIMEOUT) is checked
// end to end without hanging or faulting a GPU.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

// One thread waits, with the given limit, on a barrier whose phase can never
// complete (its count is 1 and nobody arrives).
__global__ void wait_probe_kernel(unsigned long long limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    mbar_wait(&bar, 0, &abort_flag, status, 9100, limit_ns);
  }
}

}  // namespace

cudaError_t launch_wait_probe(unsigned long long limit_ns, int* status, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace fa
