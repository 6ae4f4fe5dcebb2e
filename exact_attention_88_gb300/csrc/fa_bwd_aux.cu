// Memory-bound step ahead of the backward kernels:
//   preprocess : D_i = sum_c dO_ic * O_ic (fp32)
// It also zeroes the work counter of the backward kernel that follows it on
// the stream (when the call has one).
// It streams O and dO once with 16-byte accesses.  A block covers kUnroll
// slabs of consecutive rows and issues every load of its rows before it
// reduces any, so that each thread keeps 2 kUnroll loads in flight (one load
// at a time per thread left the kernel at about half of the copy bandwidth on
// short sequences, where a few dependent round trips are the whole kernel).
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kPreThreads = 256;
constexpr int kUnroll = 4;

// One group of d/8 consecutive lanes per row; lane g of the group handles
// columns [8g, 8g+8).  Row r of the [B, H, N] row space is (b, h, n) with
// r = (b*H + h)*N + n; O and dO may have any layout (strides), D is dense.
// Block x covers rows [x R kUnroll, (x+1) R kUnroll), R = 256 / (d/8) rows
// per slab; every lane of a group takes the same rows, so the shuffle groups
// stay converged.  O is not read again (streaming loads); dO is, by the
// backward kernels.
template <int D, bool kDense>
__global__ void __launch_bounds__(kPreThreads) bwd_preprocess_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
    float* __restrict__ Dout, long long rows, int H, int N, Layout lo, Layout ldo, int* sched) {
  constexpr int G = D / 8;                  // lanes per row (8 or 16)
  pdl_wait();  // the kernel ahead on the stream (the forward) is done
  pdl_launch_dependents();
  if (sched && blockIdx.x == 0 && threadIdx.x == 0) *sched = 0;
  constexpr int R = kPreThreads / G;        // rows per slab
  const int g = threadIdx.x % G;
  const long long row0 = (long long)blockIdx.x * R * kUnroll + threadIdx.x / G;
  uint4 a[kUnroll], c[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const long long row = row0 + (long long)u * R;
    a[u] = c[u] = make_uint4(0u, 0u, 0u, 0u);
    if (row < rows) {
      long long off_o = row * D, off_do = row * D;
      if constexpr (!kDense) {
        const int bh = (int)(row / N);
        const int n = (int)(row - (long long)bh * N);
        const int b = bh / H, h = bh - b * H;
        off_o = row_offset(lo, b, h, n);
        off_do = row_offset(ldo, b, h, n);
      }
      a[u] = __ldcs(reinterpret_cast<const uint4*>(o + off_o) + g);
      c[u] = __ldg(reinterpret_cast<const uint4*>(dO + off_do) + g);
    }
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
    const __nv_bfloat162* pc = reinterpret_cast<const __nv_bfloat162*>(&c[u]);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa = __bfloat1622float2(pa[e]);
      const float2 fc = __bfloat1622float2(pc[e]);
      acc = fmaf(fa.x, fc.x, acc);
      acc = fmaf(fa.y, fc.y, acc);
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const long long row = row0 + (long long)u * R;
    if (row < rows && g == 0) Dout[row] = acc;
  }
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.B * a.H * a.N;
  const long long per_block = (long long)(kPreThreads / (a.d / 8)) * kUnroll;
  const long long blocks = (rows + per_block - 1) / per_block;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int grid = (int)blocks;
  const bool dense =
      is_dense(a.lo, a.B, a.H, a.N, a.d) && is_dense(a.ldo, a.B, a.H, a.N, a.d);
  const auto* o = static_cast<const __nv_bfloat16*>(a.o);
  const auto* dO = static_cast<const __nv_bfloat16*>(a.dO);
  auto go = [&](auto kernel) {
    return launch_pdl(kernel, dim3(grid), dim3(kPreThreads), 0, s, o, dO, a.D, rows, a.H, a.N, a.lo,
                      a.ldo, a.sched);
  };
  if (a.d == 64)
    return dense ? go(bwd_preprocess_kernel<64, true>) : go(bwd_preprocess_kernel<64, false>);
  return dense ? go(bwd_preprocess_kernel<128, true>) : go(bwd_preprocess_kernel<128, false>);
}

}  // namespace fa
