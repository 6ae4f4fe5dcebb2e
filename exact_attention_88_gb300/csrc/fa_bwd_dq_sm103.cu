// Backward pass of exact attention, dQ: the kernel that runs the CTA body of
// fa_bwd_dq.cuh on its own (fa_bwd_dq / fa_bwd_dq_ex), and its launcher.
// fa_bwd runs the same body in the combined backward kernel.
#include "fa_bwd_dq.cuh"

namespace fa {
namespace {

template <int D, bool kExtra>
__global__ void __launch_bounds__(DqCfg<D>::kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                     const DqParams p) {
  pdl_wait();
  dq_cta<D, kExtra>(tmQ, tmK, tmV, tmDO, p, blockIdx.x);
}

template <int D>
cudaError_t launch_dq_d(const BwdArgs& a, cudaStream_t s) {
  using C = DqCfg<D>;
  CUtensorMap m[4];
  if (!encode_bwd_maps(a, m)) return cudaErrorInvalidValue;
  const DqParams p = make_dq_params(a);
  auto kernel = (a.drop.t || a.bias) ? fa_bwd_dq_kernel<D, true> : fa_bwd_dq_kernel<D, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(p.T * p.BH), dim3(C::kThreads), C::kSmem, s, m[0], m[1], m[2], m[3],
                    p);
}

}  // namespace

cudaError_t launch_bwd_dq_bf16(const BwdArgs& a, cudaStream_t s) {
  if (a.d == 64 && !a.drop.t && !a.bias) return launch_bwd_dq64_bf16(a, s);
  return a.d == 64 ? launch_dq_d<64>(a, s) : launch_dq_d<128>(a, s);
}

}  // namespace fa
