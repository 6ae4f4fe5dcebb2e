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

// Element strides of a [B, H, N, d] tensor whose d elements per row are
// contiguous: element (b, h, n, c) of layout l sits at base + b*l.b + h*l.h +
// n*l.n + c.
struct Layout {
  long long b, h, n;
};

inline Layout dense_layout(int H, int N, int d) {
  return Layout{(long long)H * N * d, (long long)N * d, (long long)d};
}

// True when l addresses a [B, H, N, d] tensor exactly as the dense layout
// does (the strides of size-1 dimensions never matter).
inline bool is_dense(const Layout& l, int B, int H, int N, int d) {
  return (B == 1 || l.b == (long long)H * N * d) && (H == 1 || l.h == (long long)N * d) &&
         (N == 1 || l.n == d);
}

// Offset in elements of row n of head (b, h).
__host__ __device__ inline long long row_offset(const Layout& l, int b, int h, int n) {
  return (long long)b * l.b + (long long)h * l.h + (long long)n * l.n;
}

// Dropout of one launch (the generator and the counter layout are described
// with philox4x32_10 in fa_common.cuh).
struct DropParams {
  uint32_t t;       // 16-bit drop threshold; 0: no dropout
  uint32_t k0, k1;  // key: seed low, seed high
  uint32_t offset;  // fourth counter word
  float rp;         // 65536 / (65536 - t): scale of the kept probabilities
};

// Everything a forward launch needs.  Pointers are device pointers.
struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;  // dense fp32 [B,H,N]
  Layout lq, lk, lv, lo;
  DropParams drop;
  const float* bias;  // additive score bias (nullptr: none), strides lb
  Layout lb;
  int B, H, N, d;
  float scale;
  int causal;
  int mask_kind;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  const int32_t* tile_order;  // block-sparse work order (nullptr: the default order)
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
  int* sched;  // work counter of the persistent backward (in the workspace), or nullptr
  void* dq;
  void* dk;
  void* dv;
  Layout lq, lk, lv, lo, ldo, ldq, ldk, ldv;
  DropParams drop;
  const float* bias;
  Layout lb;
  int B, H, N, d;
  float scale;
  int causal;
  int mask_kind;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  const int32_t* tile_order;  // block-sparse work order (nullptr: the default order)
  int* status;
};

// Encodes a 4-D TMA descriptor over a [B, H, N, d] bf16 tensor with layout
// l: x = column (d), y = row (N), then head and batch element; box = 64
// columns x box_rows rows x 1 x 1, 128-byte swizzle, out-of-range rows read
// as zero.
bool encode_bhnd_map(CUtensorMap* map, const void* base, const Layout& l, int B, int H, int N,
                     int d, int box_rows);

// The four maps every backward kernel reads (Q, K, V, dO; box 128 rows), in
// that order; false when one cannot be encoded.
bool encode_bwd_maps(const BwdArgs& a, CUtensorMap m[4]);

// Device address of the status block of the current device (no allocation:
// it is a __device__ variable), or nullptr on failure.
int* device_status();

// Streaming multiprocessors of the current device (0 when the query fails),
// looked up once per device.
int device_sm_count();

// Launch with programmatic stream serialization: the kernel's CTAs may become
// resident while the kernel ahead of it on the stream finishes; the kernel
// waits for that one (pdl_wait) before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Launchers (return the launch's cudaError_t).
cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_fwd64_bf16(const FwdArgs& a, cudaStream_t s);  // d = 64, plain
cudaError_t launch_fwd128s_bf16(const FwdArgs& a, cudaStream_t s);  // d = 128, plain
cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dkdv_bf16(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dkdv64_bf16(const BwdArgs& a, cudaStream_t s);  // d = 64, plain
cudaError_t launch_bwd_dq_bf16(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dq64_bf16(const BwdArgs& a, cudaStream_t s);  // d = 64, plain
cudaError_t launch_bwd_pair_bf16(const BwdArgs& a, cudaStream_t s);  // dK/dV and dQ, one launch
cudaError_t launch_fwd_fp32(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_fp32(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_wait_probe(unsigned long long limit_ns, int* status, cudaStream_t s);

// Block-sparse work order (query tiles, then key tiles, each most work first)
// of a T x T tile mask: tile_order_len(T) int32.
constexpr int kMaxTileOrder = 4096;  // = the largest block-mask side the kernels accept
int tile_order_len(int T);           // 0 when T is out of range
cudaError_t launch_tile_order(const uint8_t* block_mask, int T, int causal, int32_t* out,
                              cudaStream_t s);
inline int tiles_of(int n, int t) { return (n + t - 1) / t; }

// Heads per group of the kernels' grid order.  Eight heads' tiles stay in L2
// while their CTAs run.  A causal call whose four inputs (Q, K, V and dO or O,
// bf16) take at most half of the 129 MB L2 anyway gets one group of all heads:
// every head's heaviest tiles then start first instead of only the first
// group's (at N = 1024 the grouped order left 13 % of the backward to its
// tail).  Without causal masking a head's tiles carry equal work, and the
// grouped order measured as fast or faster.
inline int grid_group_heads(int B, int H, int N, int d, int causal) {
  const long long bytes = 4ll * B * H * N * d * 2;
  return (causal && bytes <= (64ll << 20)) ? B * H : 8;
}

// The argument checks of fa_bwd / fa_bwd_ex (bf16), in the same order, short
// of the workspace: host-only, no CUDA runtime call.
fa_status check_bwd_args(const void* q, const void* k, const void* v, const void* o,
                         const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale, int causal, const fa_mask* mask);

// Validates a dropout request (esize: 2 for bf16, 4 for fp32) and derives the
// kernels' parameters; no request, or a threshold of 0, is no dropout.
fa_status check_dropout(const fa_dropout* dr, int esize, DropParams* out);

// Maps a CUDA error to the ABI's status, remembering its text for
// fa_last_cuda_error() (cudaSuccess: FA_OK).
fa_status cuda_status(cudaError_t e);

}  // namespace fa
