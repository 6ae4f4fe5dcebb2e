// fp32 attention on the CUDA cores, for small fp32 workloads where tensor
// cores (bf16/tf32 inputs) would not meet fp32 accuracy.
//
// Forward: the tiled one-pass recurrence of the blog review "From Online
// Softmax to FlashAttention" ("Algorithm FlashAttention (Tiling)") with tiles
// of 32 keys staged in shared memory.  Backward: P recomputed from lse
// (summary page "FlashAttention: ...", "Key ideas: recomputation in the
// backward pass") and the textbook gradient formulas, one kernel per
// gradient side so that no atomics are needed:
//   dq kernel  (a query row per 4 threads): D_i = dO_i . O_i,
//              dQ_i = scale sum_j P_ij (dO_i . v_j - D_i) k_j
//   dkdv kernel (a key row per 4 threads): dV_j = sum_i P_ij dO_i,
//              dK_j = scale sum_i P_ij (dO_i . v_j - D_i) q_i
// Four consecutive threads share a row; thread `part` holds columns
// part, part+4, part+8, ... and dot products are summed across the four.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kRowsPerBlock = 32;
constexpr int kTileKeys = 32;

struct F32Params {
  const float* q;
  const float* k;
  const float* v;
  const float* o;
  const float* dO;
  const float* lse;
  float* out_o;
  float* out_lse;
  float* Dvec;
  float* dq;
  float* dk;
  float* dv;
  Layout lq, lk, lv, lo, ldo, ldq, ldk, ldv;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  int H, N, T;
  float scale;
  int causal;
};

__device__ __forceinline__ bool visible(const F32Params& p, int kv_limit, int i, int j) {
  if (j >= kv_limit) return false;
  if (p.causal && j > i) return false;
  if (p.block_mask && p.block_mask[(size_t)(i >> 7) * p.T + (j >> 7)] == 0) return false;
  return true;
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

template <int D>
__global__ void __launch_bounds__(128) fwd_fp32_kernel(const F32Params p) {
  constexpr int E = D / 4;
  __shared__ float sK[kTileKeys][D], sV[kTileKeys][D];
  const int bh = blockIdx.y, b = bh / p.H;
  const int part = threadIdx.x & 3;
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 2);
  const size_t head = (size_t)bh * p.N;  // lse and D rows (dense)
  const int hd = bh - b * p.H;
  const float* qh = p.q + row_offset(p.lq, b, hd, 0);
  const float* kh = p.k + row_offset(p.lk, b, hd, 0);
  const float* vh = p.v + row_offset(p.lv, b, hd, 0);
  float* ooh = p.out_o + row_offset(p.lo, b, hd, 0);
  const int kv_limit = p.kv_len ? max(0, min(p.kv_len[b], p.N)) : p.N;
  float qr[E], acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    qr[e] = row < p.N ? qh[(long long)row * p.lq.n + 4 * e + part] : 0.f;
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j0 = 0; j0 < kv_limit; j0 += kTileKeys) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTileKeys * D; idx += blockDim.x) {
      const int jj = idx / D, c = idx % D, j = j0 + jj;
      sK[jj][c] = j < p.N ? kh[(long long)j * p.lk.n + c] : 0.f;
      sV[jj][c] = j < p.N ? vh[(long long)j * p.lv.n + c] : 0.f;
    }
    __syncthreads();
    float s[kTileKeys];
    float tmax = -INFINITY;
#pragma unroll 4
    for (int jj = 0; jj < kTileKeys; ++jj) {
      float part_dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) part_dot = fmaf(qr[e], sK[jj][4 * e + part], part_dot);
      const float x = quad_sum(part_dot) * p.scale;
      s[jj] = (row < p.N && visible(p, kv_limit, row, j0 + jj)) ? x : -INFINITY;
      tmax = fmaxf(tmax, s[jj]);
    }
    const float m_new = fmaxf(m, tmax);
    if (m_new == -INFINITY) continue;  // nothing visible yet
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    l *= alpha;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= alpha;
#pragma unroll 4
    for (int jj = 0; jj < kTileKeys; ++jj) {
      const float pj = expf(s[jj] - m_new);
      l += pj;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(pj, sV[jj][4 * e + part], acc[e]);
    }
    m = m_new;
  }
  if (row < p.N) {
    const bool empty = !(l > 0.f);
    const float inv = empty ? 0.f : 1.f / l;
#pragma unroll
    for (int e = 0; e < E; ++e) ooh[(long long)row * p.lo.n + 4 * e + part] = acc[e] * inv;
    if (part == 0) p.out_lse[head + row] = empty ? -INFINITY : m + logf(l);
  }
}

template <int D>
__global__ void __launch_bounds__(128) bwd_fp32_dq_kernel(const F32Params p) {
  constexpr int E = D / 4;
  __shared__ float sK[kTileKeys][D], sV[kTileKeys][D];
  const int bh = blockIdx.y, b = bh / p.H;
  const int part = threadIdx.x & 3;
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 2);
  const size_t head = (size_t)bh * p.N;  // lse and D rows (dense)
  const int hd = bh - b * p.H;
  const float* qh = p.q + row_offset(p.lq, b, hd, 0);
  const float* kh = p.k + row_offset(p.lk, b, hd, 0);
  const float* vh = p.v + row_offset(p.lv, b, hd, 0);
  const float* oh = p.o + row_offset(p.lo, b, hd, 0);
  const float* doh = p.dO + row_offset(p.ldo, b, hd, 0);
  float* dqh = p.dq + row_offset(p.ldq, b, hd, 0);
  const int kv_limit = p.kv_len ? max(0, min(p.kv_len[b], p.N)) : p.N;
  float qr[E], dor[E], g[E];
  float dd = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const bool in = row < p.N;
    qr[e] = in ? qh[(long long)row * p.lq.n + 4 * e + part] : 0.f;
    dor[e] = in ? doh[(long long)row * p.ldo.n + 4 * e + part] : 0.f;
    dd = fmaf(dor[e], in ? oh[(long long)row * p.lo.n + 4 * e + part] : 0.f, dd);
    g[e] = 0.f;
  }
  dd = quad_sum(dd);
  const float lse = row < p.N ? p.lse[head + row] : -INFINITY;
  if (row < p.N && part == 0) p.Dvec[head + row] = dd;
  for (int j0 = 0; j0 < kv_limit; j0 += kTileKeys) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTileKeys * D; idx += blockDim.x) {
      const int jj = idx / D, c = idx % D, j = j0 + jj;
      sK[jj][c] = j < p.N ? kh[(long long)j * p.lk.n + c] : 0.f;
      sV[jj][c] = j < p.N ? vh[(long long)j * p.lv.n + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 2
    for (int jj = 0; jj < kTileKeys; ++jj) {
      float sd = 0.f, pd = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        sd = fmaf(qr[e], sK[jj][4 * e + part], sd);
        pd = fmaf(dor[e], sV[jj][4 * e + part], pd);
      }
      sd = quad_sum(sd);
      pd = quad_sum(pd);
      const bool vis = row < p.N && lse != -INFINITY && visible(p, kv_limit, row, j0 + jj);
      const float pij = vis ? expf(sd * p.scale - lse) : 0.f;
      const float ds = pij * (pd - dd);
#pragma unroll
      for (int e = 0; e < E; ++e) g[e] = fmaf(ds, sK[jj][4 * e + part], g[e]);
    }
  }
  if (row < p.N) {
#pragma unroll
    for (int e = 0; e < E; ++e) dqh[(long long)row * p.ldq.n + 4 * e + part] = g[e] * p.scale;
  }
}

template <int D>
__global__ void __launch_bounds__(128) bwd_fp32_dkdv_kernel(const F32Params p) {
  constexpr int E = D / 4;
  __shared__ float sQ[kTileKeys][D], sDO[kTileKeys][D], sL[kTileKeys], sDd[kTileKeys];
  const int bh = blockIdx.y, b = bh / p.H;
  const int part = threadIdx.x & 3;
  const int key = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 2);
  const size_t head = (size_t)bh * p.N;  // lse and D rows (dense)
  const int hd = bh - b * p.H;
  const float* qh = p.q + row_offset(p.lq, b, hd, 0);
  const float* kh = p.k + row_offset(p.lk, b, hd, 0);
  const float* vh = p.v + row_offset(p.lv, b, hd, 0);
  const float* doh = p.dO + row_offset(p.ldo, b, hd, 0);
  float* dkh = p.dk + row_offset(p.ldk, b, hd, 0);
  float* dvh = p.dv + row_offset(p.ldv, b, hd, 0);
  const int kv_limit = p.kv_len ? max(0, min(p.kv_len[b], p.N)) : p.N;
  float kr[E], vr[E], gk[E], gv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const bool in = key < p.N;
    kr[e] = in ? kh[(long long)key * p.lk.n + 4 * e + part] : 0.f;
    vr[e] = in ? vh[(long long)key * p.lv.n + 4 * e + part] : 0.f;
    gk[e] = gv[e] = 0.f;
  }
  for (int i0 = 0; i0 < p.N; i0 += kTileKeys) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTileKeys * D; idx += blockDim.x) {
      const int ii = idx / D, c = idx % D, i = i0 + ii;
      sQ[ii][c] = i < p.N ? qh[(long long)i * p.lq.n + c] : 0.f;
      sDO[ii][c] = i < p.N ? doh[(long long)i * p.ldo.n + c] : 0.f;
    }
    if (threadIdx.x < kTileKeys) {
      const int i = i0 + threadIdx.x;
      sL[threadIdx.x] = i < p.N ? p.lse[head + i] : -INFINITY;
      sDd[threadIdx.x] = i < p.N ? p.Dvec[head + i] : 0.f;
    }
    __syncthreads();
#pragma unroll 2
    for (int ii = 0; ii < kTileKeys; ++ii) {
      float sd = 0.f, pd = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        sd = fmaf(kr[e], sQ[ii][4 * e + part], sd);
        pd = fmaf(vr[e], sDO[ii][4 * e + part], pd);
      }
      sd = quad_sum(sd);
      pd = quad_sum(pd);
      const int i = i0 + ii;
      const bool vis = key < p.N && i < p.N && sL[ii] != -INFINITY && visible(p, kv_limit, i, key);
      const float pij = vis ? expf(sd * p.scale - sL[ii]) : 0.f;
      const float ds = pij * (pd - sDd[ii]);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        gv[e] = fmaf(pij, sDO[ii][4 * e + part], gv[e]);
        gk[e] = fmaf(ds, sQ[ii][4 * e + part], gk[e]);
      }
    }
  }
  if (key < p.N) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      dkh[(long long)key * p.ldk.n + 4 * e + part] = gk[e] * p.scale;
      dvh[(long long)key * p.ldv.n + 4 * e + part] = gv[e];
    }
  }
}

F32Params common(int H, int N, float scale, int causal, int mask_kind, const int32_t* kv,
                 const uint8_t* bm) {
  F32Params p{};
  p.H = H;
  p.N = N;
  p.T = tiles_of(N, 128);
  p.scale = scale;
  p.causal = causal;
  p.kv_len = mask_kind == FA_MASK_KEY_PADDING ? kv : nullptr;
  p.block_mask = mask_kind == FA_MASK_BLOCK_SPARSE ? bm : nullptr;
  return p;
}

}  // namespace

cudaError_t launch_fwd_fp32(const FwdArgs& a, cudaStream_t s) {
  F32Params p = common(a.H, a.N, a.scale, a.causal, a.mask_kind, a.kv_len, a.block_mask);
  p.q = static_cast<const float*>(a.q);
  p.k = static_cast<const float*>(a.k);
  p.v = static_cast<const float*>(a.v);
  p.out_o = static_cast<float*>(a.o);
  p.out_lse = a.lse;
  p.lq = a.lq;
  p.lk = a.lk;
  p.lv = a.lv;
  p.lo = a.lo;
  dim3 grid(tiles_of(a.N, kRowsPerBlock), a.B * a.H);
  if (a.d == 64)
    fwd_fp32_kernel<64><<<grid, 128, 0, s>>>(p);
  else
    fwd_fp32_kernel<128><<<grid, 128, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_fp32(const BwdArgs& a, cudaStream_t s) {
  F32Params p = common(a.H, a.N, a.scale, a.causal, a.mask_kind, a.kv_len, a.block_mask);
  p.q = static_cast<const float*>(a.q);
  p.k = static_cast<const float*>(a.k);
  p.v = static_cast<const float*>(a.v);
  p.o = static_cast<const float*>(a.o);
  p.dO = static_cast<const float*>(a.dO);
  p.lse = a.lse;
  p.Dvec = a.D;
  p.dq = static_cast<float*>(a.dq);
  p.dk = static_cast<float*>(a.dk);
  p.dv = static_cast<float*>(a.dv);
  p.lq = a.lq;
  p.lk = a.lk;
  p.lv = a.lv;
  p.lo = a.lo;
  p.ldo = a.ldo;
  p.ldq = a.ldq;
  p.ldk = a.ldk;
  p.ldv = a.ldv;
  dim3 grid(tiles_of(a.N, kRowsPerBlock), a.B * a.H);
  if (a.d == 64) {
    bwd_fp32_dq_kernel<64><<<grid, 128, 0, s>>>(p);
    bwd_fp32_dkdv_kernel<64><<<grid, 128, 0, s>>>(p);
  } else {
    bwd_fp32_dq_kernel<128><<<grid, 128, 0, s>>>(p);
    bwd_fp32_dkdv_kernel<128><<<grid, 128, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace fa
