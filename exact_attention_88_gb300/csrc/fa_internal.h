// Host-side plumbing shared by the translation units of libfa: argument
// bundles handed to the kernel launchers, TMA descriptor encoding and the
// per-device status block.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "fa.h"

namespace fa {

// Code the kernels write into status[0] when a wait gives up (FA_ERR_TIMEOUT).
constexpr int kStatusTimeoutCode = 6;

// Everything a forward launch needs.  Pointers are device pointers.
struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, N, d;
  float scale;
  int causal;
  int mask_kind;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  int* status;  // 4-int device status block
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dO;
  const float* lse;
  float* D;  // fp32 [B,H,N]
  void* dq;
  void* dk;
  void* dv;
  int B, H, N, d;
  float scale;
  int causal;
  int mask_kind;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  int* status;
};

// Encodes a 3-D TMA descriptor over a [BH, N, d] bf16 tensor: x = column
// (d), y = row (N), z = head; box = 64 columns x box_rows rows x 1 head,
// 128-byte swizzle, out-of-range rows read as zero.
bool encode_bhnd_map(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows);

// Device address of the status block of the current device (no allocation:
// it is a __device__ variable), or nullptr on failure.
int* device_status();

// Launchers (return the launch's cudaError_t).
cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dkdv_bf16(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dq_bf16(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_fwd_fp32(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_fp32(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_umma_probe(const void* a, const void* b, float* d, int M, int N, int K,
                              int a_mn, int b_mn, int a_tmem, int use_tma, int* status,
                              cudaStream_t s);
cudaError_t launch_wait_probe(unsigned long long limit_ns, int* status, cudaStream_t s);

inline int tiles_of(int n, int t) { return (n + t - 1) / t; }

}  // namespace fa
