// Backward pass of exact attention, dK / dV and dQ in one launch.  The dK/dV
// CTAs (one per key tile, fa_bwd_dkdv.cuh, fa_bwd_dkdv64.cuh) and the dQ CTAs
// (one per query tile, fa_bwd_dq.cuh, fa_bwd_dq64.cuh) read the same inputs
// and write disjoint outputs, so they can share the GPU: the combined grid
// holds the dK/dV CTAs first (the longer kind), then the dQ CTAs, each kind in
// its own order (heaviest tiles first).  The dQ CTAs thus fill the SMs that the
// last dK/dV CTAs leave idle, from a single launch on the caller's stream.  (Run
// side by side from the start, the two kinds stream Q, dO and K, V of a group of
// heads at once, about the size of L2, and the pair took 1.5 times as long.)
// The two bodies of a pair have the same
// thread count, TMEM allocation and CTAs per SM; the dynamic shared memory is
// the larger of the two.
// At d = 128 without a block mask, key padding, dropout or a bias, the dQ
// part is one persistent CTA per SM that takes query tiles one after another
// (fa_bwd_persist.cuh): long causal 2.525 against 2.552-2.562 ms.
#include "fa_bwd_dkdv.cuh"
#include "fa_bwd_dkdv64.cuh"
#include "fa_bwd_dq.cuh"
#include "fa_bwd_dq64.cuh"
#include "fa_bwd_persist.cuh"

namespace fa {
namespace {

static_assert(BwdCfg<64>::kThreads == DqCfg<64>::kThreads &&
                  BwdCfg<128>::kThreads == DqCfg<128>::kThreads,
              "the dK/dV and dQ CTAs of a pair run with the same block size");
static_assert(Bwd64Cfg::kThreads == Dq64Cfg::kThreads,
              "the dK/dV and dQ CTAs of a pair run with the same block size");

// CTA lin of the combined grid -> kind (0: dK/dV, 1: dQ) and the CTA's index in
// that kind's own grid of n0 CTAs (dK/dV, first) or n1 (dQ).
__device__ __forceinline__ void split_grid(int lin, int n0, int n1, int* kind, int* idx) {
  (void)n1;
  *kind = lin < n0 ? 0 : 1;
  *idx = lin < n0 ? lin : lin - n0;
}

template <int D, bool kExtra>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const BwdParams pk, const DqParams pq) {
  pdl_wait();
  int kind, idx;
  split_grid(blockIdx.x, pk.T * pk.BH, pq.T * pq.BH, &kind, &idx);
  if (kind == 0)
    dkdv_cta<D, kExtra>(tmQ, tmK, tmV, tmDO, pk, idx);
  else
    dq_cta<D, kExtra>(tmQ, tmK, tmV, tmDO, pq, idx);
}

__global__ void __launch_bounds__(Bwd64Cfg::kThreads, 2)
    fa_bwd64_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const Bwd64Params pk, const Dq64Params pq) {
  pdl_wait();
  int kind, idx;
  split_grid(blockIdx.x, pk.T * pk.BH, pq.T * pq.BH, &kind, &idx);
  if (kind == 0)
    dkdv64_cta(tmQ, tmK, tmV, tmDO, pk, idx);
  else
    dq64_cta(tmQ, tmK, tmV, tmDO, pq, idx);
}

// Persistent dQ: the first n0 CTAs are the one-per-unit dK/dV CTAs; the last
// gridDim - n0 CTAs each hold 512 TMEM columns and take dQ units from the
// counter (CTA x starts with unit x) until none is left.
template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                          const BwdParams pk, const DqParams pq, int* counter) {
  pdl_wait();
  const int n0 = pk.T * pk.BH, n = n0 + pq.T * pq.BH;
  if ((int)blockIdx.x < n0) {
    dkdv_cta<D, false>(tmQ, tmK, tmV, tmDO, pk, blockIdx.x);
    return;
  }
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5;
  if (warp == BwdCfg<D>::kMathWarps + 1) tmem_alloc(&tmem_slot, BwdCfg<D>::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  pdl_launch_dependents();  // TMEM held: the next kernel may become resident
  dq_persist<D>(tmQ, tmK, tmV, tmDO, pq, tmem, blockIdx.x, n0, n, counter);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == BwdCfg<D>::kMathWarps + 1) {
    __syncwarp();
    tmem_dealloc(tmem, BwdCfg<D>::kTmemCols);
  }
}

template <class Kernel, class PK, class PQ>
cudaError_t launch_pair(Kernel kernel, int threads, int smem, const CUtensorMap* m, const PK& pk,
                        const PQ& pq, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(pk.T * pk.BH + pq.T * pq.BH), dim3(threads), smem, s, m[0], m[1],
                    m[2], m[3], pk, pq);
}

template <int D>
cudaError_t launch_pair_d(const BwdArgs& a, const CUtensorMap* m, cudaStream_t s) {
  const int smem = max(BwdCfg<D>::kSmem, DqCfg<D>::kSmem);
  auto kernel = (a.drop.t || a.bias) ? fa_bwd_pair_kernel<D, true> : fa_bwd_pair_kernel<D, false>;
  return launch_pair(kernel, BwdCfg<D>::kThreads, smem, m, make_dkdv_params(a), make_dq_params(a), s);
}

}  // namespace

cudaError_t launch_bwd_pair_bf16(const BwdArgs& a, cudaStream_t s) {
  CUtensorMap m[4];
  if (!encode_bwd_maps(a, m)) return cudaErrorInvalidValue;
  if (a.d == 128 && !a.drop.t && !a.bias && a.mask_kind == FA_MASK_NONE && a.sched) {
    const BwdParams pk = make_dkdv_params(a);
    const DqParams pq = make_dq_params(a);
    const int units = pk.T * pk.BH + pq.T * pq.BH;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int smem = max(BwdCfg<128>::kSmem, DqCfg<128>::kSmem);
    auto kernel = fa_bwd_persist_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int n0 = pk.T * pk.BH;
    return launch_pdl(kernel, dim3(n0 + min(units - n0, sms)), dim3(BwdCfg<128>::kThreads), smem, s,
                      m[0], m[1], m[2], m[3], pk, pq, a.sched);
  }
  if (a.d == 64 && !a.drop.t && !a.bias)
    return launch_pair(fa_bwd64_pair_kernel, Bwd64Cfg::kThreads, max(Bwd64Cfg::kSmem, Dq64Cfg::kSmem),
                       m, make_dkdv64_params(a), make_dq64_params(a), s);
  return a.d == 64 ? launch_pair_d<64>(a, m, s) : launch_pair_d<128>(a, m, s);
}

}  // namespace fa
