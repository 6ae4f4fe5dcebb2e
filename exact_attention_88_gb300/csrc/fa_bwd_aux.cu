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
// columns [8g, 8g+8).  Row r of the [B, H, N] row space is (b, h, n) with
// r = (b*H + h)*N + n; O and dO may have any layout (strides), D is dense.
template <int D, bool kDense>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                             const __nv_bfloat16* __restrict__ dO,
                                                             float* __restrict__ Dout,
                                                             long long rows, int H, int N,
                                                             Layout lo, Layout ldo) {
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
      long long off_o = row * D, off_do = row * D;
      if constexpr (!kDense) {
        const int bh = (int)(row / N);
        const int n = (int)(row - (long long)bh * N);
        const int b = bh / H, h = bh - b * H;
        off_o = row_offset(lo, b, h, n);
        off_do = row_offset(ldo, b, h, n);
      }
      const uint4 a = reinterpret_cast<const uint4*>(o + off_o)[g];
      const uint4 c = reinterpret_cast<const uint4*>(dO + off_do)[g];
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* pc = reinterpret_cast<const __nv_bfloat162*>(&c);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(pa[e]);
        const float2 fc = __bfloat1622float2(pc[e]);
        acc = fmaf(fa.x, fc.x, acc);
        acc = fmaf(fa.y, fc.y, acc);
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
  const bool dense =
      is_dense(a.lo, a.B, a.H, a.N, a.d) && is_dense(a.ldo, a.B, a.H, a.N, a.d);
  const auto* o = static_cast<const __nv_bfloat16*>(a.o);
  const auto* dO = static_cast<const __nv_bfloat16*>(a.dO);
  auto go = [&](auto kernel) {
    kernel<<<grid, threads, 0, s>>>(o, dO, a.D, rows, a.H, a.N, a.lo, a.ldo);
  };
  if (a.d == 64)
    dense ? go(bwd_preprocess_kernel<64, true>) : go(bwd_preprocess_kernel<64, false>);
  else
    dense ? go(bwd_preprocess_kernel<128, true>) : go(bwd_preprocess_kernel<128, false>);
  return cudaGetLastError();
}

}  // namespace fa
