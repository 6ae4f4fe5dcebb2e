// Work order of a block-sparse mask: the tiles of each kind sorted by the
// work each carries, most first, so that a grid that gives one CTA per tile
// row (forward, dQ) or per tile column (dK/dV) starts its longest CTAs first
// instead of ending with them.
// The order changes only which CTA takes which tile, never what a tile
// computes ("FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness", summary page, "Extension: block-sparse FlashAttention": the
// kernels visit only the nonzero blocks of the mask).
//
// One CTA: its warps read the mask by rows (lanes on consecutive 16-byte
// chunks where the rows allow it, eight loads in flight per warp) and count
// each row's visible tiles (causal: key tile <= query tile) with a warp
// reduction and each column's in shared memory; then a stable counting sort of
// each kind by its counts writes every tile at its rank: the number of tiles
// with more work, plus those with as much and a lower index.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kOrderThreads = 512;

// Writes out[r] = e for e in [0, n), r = e's rank in c: elements with a larger
// count, then those with the same count and a lower index, come first (a
// stable counting sort, counts in [0, V]).  hist: V + 1 ints of shared memory.
// Called by the whole CTA.
__device__ void place_by_count(const int* c, int n, int V, int* hist, int32_t* out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  const int nb = V + 1;
  for (int v = tid; v < nb; v += nthr) hist[v] = 0;
  __syncthreads();
  // one atomic per distinct count in a warp (tiles of a regular pattern share
  // one count, and atomics on one address serialize)
  for (int base = 0; base < n; base += nthr) {
    const int e = base + tid;
    const int v = e < n ? c[e] : -1;
    const unsigned same = __match_any_sync(0xffffffffu, v);
    if (v >= 0 && (same & ((1u << lane) - 1u)) == 0u) atomicAdd(&hist[v], __popc(same));
  }
  __syncthreads();
  // hist[v] := elements with a count above v (a suffix sum over the bins):
  // each thread owns a run of bins; the runs above its own are summed by a
  // block-wide scan of the run totals
  const int per = (nb + nthr - 1) / nthr;
  const int lo = min(tid * per, nb), hi = min(lo + per, nb);
  int own = 0;
  for (int v = lo; v < hi; ++v) own += hist[v];
  int incl = own;  // inclusive prefix of the run totals, in thread order
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  __shared__ int warp_total[32], grand;
  if (lane == 31) warp_total[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = nthr >> 5;
    int t = lane < nw ? warp_total[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += x;
    }
    if (lane < nw) warp_total[lane] = t;  // inclusive over warps
    if (lane == 31) grand = t;
  }
  __syncthreads();
  if (warp > 0) incl += warp_total[warp - 1];
  int above = grand - incl;  // elements in the runs of higher threads
  for (int v = hi - 1; v >= lo; --v) {
    const int h = hist[v];
    hist[v] = above;
    above += h;
  }
  __syncthreads();
  // stable placement: chunks of the CTA's size in index order, the warps of a
  // chunk one after another; equal counts within a warp by lane order
  for (int base = 0; base < n; base += nthr) {
    const int e = base + tid;
    const bool valid = e < n;
    const int v = valid ? c[e] : -1;
    const unsigned same = __match_any_sync(0xffffffffu, v);
    const int before = __popc(same & ((1u << lane) - 1u));
    const int nw = (min(n - base, nthr) + 31) >> 5;
    for (int w = 0; w < nw; ++w) {
      if (warp == w && valid) {
        out[hist[v] + before] = e;
        __syncwarp(same);
        if (before == 0) hist[v] += __popc(same);
      }
      __syncthreads();
    }
  }
}

template <bool kVec>
__global__ void __launch_bounds__(kOrderThreads)
    tile_order_kernel(const uint8_t* __restrict__ bm, int T, int causal, int32_t* __restrict__ out) {
  extern __shared__ int cnt[];  // rows [0, T), columns [T, 2T), bins
  pdl_wait();  // the kernel ahead on the stream is done (it may read `out`)
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int e = threadIdx.x; e < 2 * T; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  int* col = cnt + T;
  if constexpr (kVec) {
    // T % 16 == 0 and a 16-byte aligned mask: a warp owns rows warp + nwarps r
    // and takes them 512 columns (one 16-byte chunk per lane) at a time, eight
    // rows' loads in flight before it counts any; each lane keeps the counts
    // of its 16 columns in registers and adds them to shared memory once per
    // 512 columns
    constexpr int kBatch = 8;
    const int rows = warp < T ? (T - 1 - warp) / nwarps + 1 : 0;
    for (int g0 = 0; g0 < T; g0 += 512) {
      const int j0 = g0 + 16 * lane;
      int colc[16];
#pragma unroll
      for (int b = 0; b < 16; ++b) colc[b] = 0;
      for (int r0 = 0; r0 < rows; r0 += kBatch) {
        uint4 w[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int i = warp + nwarps * (r0 + u);
          w[u] = make_uint4(0u, 0u, 0u, 0u);
          if (r0 + u < rows && j0 < (causal ? i + 1 : T))
            w[u] = *reinterpret_cast<const uint4*>(bm + (size_t)i * T + j0);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (r0 + u >= rows) break;  // warp-uniform
          const int i = warp + nwarps * (r0 + u);
          const int jend = causal ? i + 1 : T;  // visible key tiles: j < jend
          const uint32_t word[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
          int c = 0;
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            const int vis = ((word[b >> 2] >> (8 * (b & 3))) & 0xffu) != 0u && j0 + b < jend;
            c += vis;
            colc[b] += vis;
          }
          c = __reduce_add_sync(0xffffffffu, c);
          if (lane == 0 && c != 0) atomicAdd(&cnt[i], c);
        }
      }
#pragma unroll
      for (int b = 0; b < 16; ++b)
        if (colc[b] != 0) atomicAdd(&col[j0 + b], colc[b]);  // nonzero: j0 + b < T
    }
  } else {
    for (int i = warp; i < T; i += nwarps) {
      const uint8_t* row = bm + (size_t)i * T;
      const int jend = causal ? i + 1 : T;
      int c = 0;
      for (int j = lane; j < jend; j += 32) {
        if (row[j] != 0) {
          ++c;
          atomicAdd(&col[j], 1);
        }
      }
      c = __reduce_add_sync(0xffffffffu, c);
      if (lane == 0) cnt[i] = c;
    }
  }
  __syncthreads();
  // every count is in shared memory: the output may now be overwritten
  int* hist = cnt + 2 * T;  // 2T + 2 ints
  place_by_count(cnt, T, T, hist, out);
  place_by_count(cnt + T, T, T, hist, out + T);
}

}  // namespace

int tile_order_len(int T) { return (T < 1 || T > kMaxTileOrder) ? 0 : 2 * T; }

cudaError_t launch_tile_order(const uint8_t* block_mask, int T, int causal, int32_t* out,
                              cudaStream_t s) {
  // counts (2T ints) and the counting sort's bins (2T + 2 ints): <= 64 KB
  const int smem = (tile_order_len(T) + 2 * T + 2) * (int)sizeof(int);
  const bool vec = T % 16 == 0 && (reinterpret_cast<uintptr_t>(block_mask) & 15u) == 0;
  auto kernel = vec ? tile_order_kernel<true> : tile_order_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(1), dim3(kOrderThreads), (size_t)smem, s, block_mask, T, causal, out);
}

}  // namespace fa
