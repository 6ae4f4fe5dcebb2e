// Backward pass of exact attention, dK and dV: the kernel that runs the CTA
// body of fa_bwd_dkdv.cuh on its own (fa_bwd_dkdv / fa_bwd_dkdv_ex), and its
// launcher.  fa_bwd runs the same body in the combined backward kernel.
#include "fa_bwd_dkdv.cuh"

namespace fa {
namespace {

template <int D, bool kExtra>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const BwdParams p) {
  pdl_wait();
  dkdv_cta<D, kExtra>(tmQ, tmK, tmV, tmDO, p, blockIdx.x);
}

template <int D>
cudaError_t launch_dkdv_d(const BwdArgs& a, cudaStream_t s) {
  using C = BwdCfg<D>;
  CUtensorMap m[4];
  if (!encode_bwd_maps(a, m)) return cudaErrorInvalidValue;
  const BwdParams p = make_dkdv_params(a);
  auto kernel = (a.drop.t || a.bias) ? fa_bwd_dkdv_kernel<D, true> : fa_bwd_dkdv_kernel<D, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(p.T * p.BH), dim3(C::kThreads), C::kSmem, s, m[0], m[1], m[2], m[3],
                    p);
}

}  // namespace

cudaError_t launch_bwd_dkdv_bf16(const BwdArgs& a, cudaStream_t s) {
  // d = 64 calls without dropout or a bias: 64-row steps, two CTAs per SM
  if (a.d == 64 && !a.drop.t && !a.bias) return launch_bwd_dkdv64_bf16(a, s);
  return a.d == 64 ? launch_dkdv_d<64>(a, s) : launch_dkdv_d<128>(a, s);
}

}  // namespace fa
