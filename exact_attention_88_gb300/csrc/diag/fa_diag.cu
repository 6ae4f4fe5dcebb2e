// Test-only diagnostics, built into libfa_diag.so beside libfa.so and loaded
// by the tests alone; nothing here is part of libfa's C ABI.
//  * A single-CTA tensor-core GEMM, D = A B^T, that stages its operands
//    exactly the way the attention kernels do (128-byte-swizzled K-major or
//    MN-major shared-memory tiles, TMA or plain loads, A optionally in tensor
//    memory as packed bf16 pairs), so a test can confirm every operand layout
//    the kernels depend on against a host matrix product.
//  * The dropout keep mask drawn with the device code of the attention
//    kernels (fa_common.cuh), through both of its code paths, so a test can
//    compare it bit for bit with the oracle's.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

// 4-int status block of the diagnostics (its own: no allocation).
__device__ int g_diag_status[4];

constexpr int kProbeM = 128;
constexpr int kProbeSmem = 128 * 128 * 2 + 256 * 128 * 2 + 1024;  // A, B, alignment slack

__global__ void __launch_bounds__(128, 1)
    umma_probe_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ Bm,
                      float* __restrict__ Dm, int N, int K, int a_mn, int b_mn, int a_tmem,
                      int use_tma, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                        // 128 x K bf16
  uint8_t* sB = smem + kProbeM * 128 * 2;    // N x K bf16
  __shared__ uint64_t bar_load, bar_mma;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;

  if (tid == 0) {
    mbar_init(&bar_load, 1);
    mbar_init(&bar_mma, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  const int kchunks = K / 64;

  // ---- stage B (and A when it goes through shared memory) -----------------
  if (use_tma) {
    if (tid == 0) {
      uint32_t bytes = (uint32_t)N * K * 2 + (a_tmem ? 0u : (uint32_t)kProbeM * K * 2);
      mbar_expect_tx(&bar_load, bytes);
      for (int c = 0; c < kchunks; ++c) {
        if (!a_tmem) tma_load_4d(&tmA, &bar_load, sA + c * kProbeM * 128, c * 64, 0, 0, 0);
        tma_load_4d(&tmB, &bar_load, sB + c * N * 128, c * 64, 0, 0, 0);
      }
    }
  } else {
    for (int idx = tid; idx < N * K; idx += blockDim.x) {
      const int n = idx / K, k = idx % K;
      uint32_t off = b_mn ? (uint32_t)(n / 64) * (K * 128) + sw128_offset(k, n % 64)
                          : (uint32_t)(k / 64) * (N * 128) + sw128_offset(n, k % 64);
      *reinterpret_cast<__nv_bfloat16*>(sB + off) = Bm[idx];
    }
    if (!a_tmem) {
      for (int idx = tid; idx < kProbeM * K; idx += blockDim.x) {
        const int m = idx / K, k = idx % K;
        uint32_t off = a_mn ? (uint32_t)(m / 64) * (K * 128) + sw128_offset(k, m % 64)
                            : (uint32_t)(k / 64) * (kProbeM * 128) + sw128_offset(m, k % 64);
        *reinterpret_cast<__nv_bfloat16*>(sA + off) = A[idx];
      }
    }
    fence_proxy_async_smem();
  }
  // ---- A into tensor memory (columns 256..) --------------------------------
  const uint32_t a_col = 256;
  if (a_tmem) {
    const int m = tid;  // one row per thread, lane m
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int ncols = (K / 16) * 8;  // 8 columns per 16 K elements
    for (int c0 = 0; c0 < ncols; c0 += 16) {
      uint32_t r[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = c0 + j;
        const float lo = __bfloat162float(A[m * K + 2 * col]);
        const float hi = __bfloat162float(A[m * K + 2 * col + 1]);
        r[j] = pack_bf16(lo, hi);  // even k in the low half
      }
      FA_TMEM_ST16(tbase + lane_base + a_col + c0, r);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- issue the MMAs -------------------------------------------------------
  if (tid == 0) {
    bool ok = true;
    if (use_tma) ok = mbar_wait(&bar_load, 0, &abort_flag, status, 9001);
    if (ok) {
      const uint32_t idesc = idesc_bf16(kProbeM, N, a_mn != 0, b_mn != 0);
      const uint32_t a_base = smem_addr(sA), b_base = smem_addr(sB);
      for (int ks = 0; ks < K / 16; ++ks) {
        uint64_t bd = b_mn ? sdesc_sw128(b_base + ks * 2048, K * 128, 1024)
                           : sdesc_sw128(b_base + (ks / 4) * (N * 128) + (ks % 4) * 32, 16, 1024);
        if (a_tmem) {
          mma_ts(tbase, tbase + a_col + ks * 8, bd, idesc, ks > 0);
        } else {
          uint64_t ad = a_mn ? sdesc_sw128(a_base + ks * 2048, K * 128, 1024)
                             : sdesc_sw128(a_base + (ks / 4) * (kProbeM * 128) + (ks % 4) * 32, 16, 1024);
          mma_ss(tbase, ad, bd, idesc, ks > 0);
        }
      }
    }
    mma_commit(&bar_mma);  // also covers the no-MMA path: arrives at once
    if (use_tma && !ok) mbar_drain(&bar_load, 0);
  }
  __syncwarp();
  bool done = mbar_wait_warp(&bar_mma, 0, &abort_flag, status, 9002);
  tc_fence_after();
  if (done) {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int m = tid;
    for (int c0 = 0; c0 < N; c0 += 32) {
      uint32_t r[32];
      FA_TMEM_LD32_SYNC(tbase + lane_base + c0, r);
#pragma unroll
      for (int j = 0; j < 32; ++j) Dm[(size_t)m * N + c0 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tbase, 512);
  }
}

// Dropout keep mask out[bh][i][j] through the row path of the forward and dQ
// kernels: a thread per (bh, row i, 32 keys).
__global__ void dropout_mask_rowbits_kernel(uint8_t* out, int N, DropParams d) {
  const int bh = blockIdx.z, i = blockIdx.y;
  const int key0 = 32 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (key0 >= N) return;
  const uint32_t bits = keep_bits_of_row(d, (uint32_t)bh, i, key0);
  uint8_t* row = out + ((size_t)bh * N + i) * N;
  for (int c = 0; c < 32 && key0 + c < N; ++c) row[key0 + c] = (uint8_t)((bits >> c) & 1u);
}

// The same through the key path of the dK/dV kernel: each warp takes 32
// consecutive keys (a key per lane) and 32 query rows; every lane takes part
// in the shuffles, only entries inside [0, N) are written.
__global__ void dropout_mask_keys_kernel(uint8_t* out, int N, DropParams d) {
  const int bh = blockIdx.z, q0 = 32 * blockIdx.y;
  const int key = 32 * (4 * blockIdx.x + (threadIdx.x >> 5)) + (threadIdx.x & 31);
  const uint32_t bits = keep_bits_of_key(d, (uint32_t)bh, key, q0);
  if (key >= N) return;
  for (int c = 0; c < 32 && q0 + c < N; ++c)
    out[((size_t)bh * N + q0 + c) * N + key] = (uint8_t)((bits >> c) & 1u);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int* diag_status() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_diag_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

int launched(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

// D[M x N] (fp32, row-major) = A B^T on the tensor cores.  a: device bf16
// [M x K] row-major, b: device bf16 [N x K] row-major; M = 128, N in
// {64, 128, 256}, K in {64, 128}.  a_mn_major / b_mn_major stage the operand
// M/N-contiguous; a_in_tmem takes A from tensor memory (two bf16 per 32-bit
// column, even k in the low half; needs a_mn_major = 0); use_tma loads
// K-major operands with TMA.
int fa_diag_umma_gemm(const void* a, const void* b, float* d, int M, int N, int K,
                      int a_mn_major, int b_mn_major, int a_in_tmem, int use_tma, void* stream) {
  if (!a || !b || !d) return FA_ERR_INVALID_ARG;
  if (M != 128 || (N != 64 && N != 128 && N != 256) || (K != 64 && K != 128))
    return FA_ERR_UNSUPPORTED;
  if (a_in_tmem < 0 || a_in_tmem > 1 || (a_in_tmem && a_mn_major)) return FA_ERR_INVALID_ARG;
  if (use_tma && (a_mn_major || b_mn_major)) return FA_ERR_UNSUPPORTED;
  if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return FA_ERR_ALIGNMENT;
  int* st = diag_status();
  if (!st) return FA_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap ma{}, mb{};
  if (use_tma) {
    if (!encode_bhnd_map(&ma, a, dense_layout(1, kProbeM, K), 1, 1, kProbeM, K, kProbeM) ||
        !encode_bhnd_map(&mb, b, dense_layout(1, N, K), 1, 1, N, K, N))
      return FA_ERR_CUDA;
  }
  cudaError_t e = cudaFuncSetAttribute(umma_probe_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  umma_probe_kernel<<<1, 128, kProbeSmem, s>>>(ma, mb, static_cast<const __nv_bfloat16*>(a),
                                                static_cast<const __nv_bfloat16*>(b), d, N, K,
                                                a_mn_major, b_mn_major, a_in_tmem, use_tma, st);
  return launched(cudaGetLastError());
}

// The dropout keep mask Z (uint8 [B*H, N, N], 1 = kept) of `dropout`: path 0
// as the forward and dQ kernels draw it (a query row per thread, 32 keep
// bits at a time), path 1 as the dK/dV kernel does (a key per thread, the
// bits of each call shared among eight lanes).  N <= 4096.
int fa_diag_dropout_mask(uint8_t* out, int B, int H, int N, const fa_dropout* dropout, int path,
                         void* stream) {
  if (!out || !dropout) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || (long long)B * H > 65535) return FA_ERR_INVALID_ARG;
  if (N > 4096) return FA_ERR_UNSUPPORTED;
  if (path != 0 && path != 1) return FA_ERR_INVALID_ARG;
  DropParams d;
  const fa_status st = check_dropout(dropout, 2, &d);
  if (st != FA_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  if (path == 0) {
    const int chunks = (N + 31) / 32;
    dropout_mask_rowbits_kernel<<<dim3((chunks + 127) / 128, N, BH), 128, 0, s>>>(out, N, d);
  } else {
    dropout_mask_keys_kernel<<<dim3((N + 127) / 128, (N + 31) / 32, BH), 128, 0, s>>>(out, N, d);
  }
  return launched(cudaGetLastError());
}

// Synchronizes `stream`, then returns and clears the diagnostics' device
// status: 0, or 6 when a wait gave up (*site: its id).
int fa_diag_status(void* stream, int* site) {
  if (site) *site = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int* st = diag_status();
  if (!st) return FA_ERR_CUDA;
  int h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, st, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (h[0] != 0) {
    if (site) *site = h[1];
    const int z[4] = {0, 0, 0, 0};
    if (cudaMemcpy(st, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  }
  return h[0];
}

}  // extern "C"
