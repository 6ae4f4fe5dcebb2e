// Memory-bound step ahead of the backward kernels:
//   preprocess : D_i = sum_c dO_ic * O_ic (fp32)
// It streams O and dO once with 16-byte accesses; the grid is a multiple of
// the SM count and loops over the rows.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

int grid_for(long long work_items, int threads) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (work_items + threads - 1) / threads;
  long long cap = (long long)sms * 8;
  return (int)(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
}

// One group of d/8 consecutive lanes per row; lane g of the group handles
// columns [8g, 8g+8).
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint4* __restrict__ o,
                                                             const uint4* __restrict__ dO,
                                                             float* __restrict__ Dout,
                                                             long long rows) {
  constexpr int G = D / 8;  // lanes per row (8 or 16)
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const int g = threadIdx.x % G;
  // every thread runs the same number of passes so the shuffle groups stay
  // converged
  const long long groups_per_pass = nthreads / G;
  const long long passes = (rows + groups_per_pass - 1) / groups_per_pass;
  for (long long pass = 0; pass < passes; ++pass) {
    const long long row = pass * groups_per_pass + tid / G;
    float acc = 0.f;
    if (row < rows) {
      const uint4 a = o[row * G + g];
      const uint4 b = dO[row * G + g];
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(pa[e]);
        const float2 fb = __bfloat1622float2(pb[e]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && g == 0) Dout[row] = acc;
  }
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.B * a.H * a.N;
  const int threads = 256;
  const int grid = grid_for(rows * (a.d / 8), threads);
  if (a.d == 64)
    bwd_preprocess_kernel<64><<<grid, threads, 0, s>>>(
        static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dO), a.D, rows);
  else
    bwd_preprocess_kernel<128><<<grid, threads, 0, s>>>(
        static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dO), a.D, rows);
  return cudaGetLastError();
}

}  // namespace fa
