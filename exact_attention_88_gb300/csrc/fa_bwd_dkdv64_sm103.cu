// Backward pass of exact attention at d = 64, dK and dV: the kernel that runs
// the CTA body of fa_bwd_dkdv64.cuh on its own, and its launcher.  fa_bwd runs
// the same body in the combined backward kernel.
#include "fa_bwd_dkdv64.cuh"

namespace fa {
namespace {

__global__ void __launch_bounds__(Bwd64Cfg::kThreads, 2)
    fa_bwd_dkdv64_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmDO, const Bwd64Params p) {
  pdl_wait();
  dkdv64_cta(tmQ, tmK, tmV, tmDO, p, blockIdx.x);
}

}  // namespace

cudaError_t launch_bwd_dkdv64_bf16(const BwdArgs& a, cudaStream_t s) {
  using C = Bwd64Cfg;
  CUtensorMap m[4];
  if (!encode_bwd_maps(a, m)) return cudaErrorInvalidValue;
  const Bwd64Params p = make_dkdv64_params(a);
  cudaError_t e = cudaFuncSetAttribute(fa_bwd_dkdv64_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(fa_bwd_dkdv64_kernel, dim3(p.T * p.BH), dim3(C::kThreads), C::kSmem, s, m[0],
                    m[1], m[2], m[3], p);
}

}  // namespace fa
