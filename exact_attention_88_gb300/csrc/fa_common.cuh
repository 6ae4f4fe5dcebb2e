// Device-side building blocks for the sm_103a attention kernels: inline PTX
// for mbarriers, TMA tile loads, tcgen05 MMAs / TMEM traffic, shared-memory
// matrix descriptors, and bounded waits that report a timeout instead of
// hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_internal.h"

namespace fa {

constexpr float kLog2e = 1.4426950408889634f;  // scores in base 2: exp(x) = 2^(x log2 e)
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// status words.  Every kernel gets a pointer to a 4-int status block in device
// memory: [0] error code (0 = ok, 6 = timeout), [1] site id, [2] block, [3] aux.
// ---------------------------------------------------------------------------
constexpr int kStatusTimeout = 6;  // equals FA_ERR_TIMEOUT
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;     // 2 s per wait
constexpr uint64_t kDrainTimeoutNs = 500000000ull;     // 0.5 s while tearing down
constexpr uint32_t kSuspendHintNs = 200000u;           // longest sleep of one wait attempt

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report(int* status, int site) {
  if (atomicCAS(&status[0], 0, kStatusTimeout) == 0) {
    status[1] = site;
    status[2] = blockIdx.x + gridDim.x * blockIdx.y;
  }
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same with a suspend-time hint: a thread whose phase has not completed
// sleeps until it completes (or the hint runs out) instead of polling, so a
// waiting warp leaves the issue slots of its SMSP to the warps that work.
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity of `bar` has completed.  Gives up
// (returns false) when another role has already aborted, or after
// `limit_ns`, in which case it raises the CTA's abort flag and records the
// site in the status block.  Never spins without a limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, int site,
                                          uint64_t limit_ns = kWaitTimeoutNs) {
  const uint32_t a = smem_addr(bar);
  if (mbar_try(a, parity)) return true;
  const uint64_t t0 = global_timer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_sleep(a, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer() - t0 > limit_ns) {
      *abort_flag = 1;
      report(status, site);
      return false;
    }
  }
}

// Same, for all 32 lanes of a warp; the warp agrees on the outcome so that
// the .sync.aligned tcgen05 instructions that follow stay convergent.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity,
                                               volatile int* abort_flag, int* status, int site) {
  bool ok = mbar_wait(bar, parity, abort_flag, status, site);
  return __all_sync(0xffffffffu, ok);
}

// Teardown wait: ignores the abort flag, shorter limit, never reports.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  const uint64_t t0 = global_timer();
  while (!mbar_try(a, parity)) {
    if (global_timer() - t0 > kDrainTimeoutNs) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// TMA: 4-D tiled bulk tensor load into shared memory, completion counted in
// bytes on an mbarrier.  Coordinates are (x = column, y = row, h = head,
// b = batch element); the tensor map carries the three strides, so any
// layout whose d elements of a row are contiguous is read the same way.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_4d(const CUtensorMap* map, uint64_t* bar, void* dst, int x,
                                            int y, int h, int b) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(h), "r"(b)
      : "memory");
}

// TMA: bring a tile of a tensor into L2 ahead of its load (no completion
// signal; a hint that never faults on coordinates outside the tensor).
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int x, int y, int h,
                                                int b) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(h), "r"(b)
               : "memory");
}

// ---------------------------------------------------------------------------
// Block-sparse tile masks.  A CTA copies the row (or column) of the caller's
// uint8 [T, T] tile mask it walks into a shared-memory bitmap once, so that
// finding the next visible tile is a few bit scans instead of a chain of
// dependent global loads (one per skipped tile).
// ---------------------------------------------------------------------------
constexpr int kMaskBitmapWords = 128;  // tiles per bitmap: 4096 (N <= 524288)

// The block-mask bitmap of a CTA (its tile row or column).  One array per
// kernel: a kernel that runs one of several CTA bodies shares it between them.
__device__ __forceinline__ uint32_t* tile_mask_bitmap() {
  __shared__ uint32_t bits[kMaskBitmapWords];
  return bits;
}

// bits[t / 32] bit t % 32 = (first[t * stride] != 0), t < T.  Every thread of
// the CTA takes part (whole warps); a __syncthreads must follow before use.
__device__ __forceinline__ void build_tile_bitmap(uint32_t* bits, const uint8_t* first,
                                                  size_t stride, int T) {
  const int warps = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int w = warp; w < (T + 31) / 32; w += warps) {
    const int t = 32 * w + lane;
    const uint32_t on = __ballot_sync(0xffffffffu, t < T && first[(size_t)t * stride] != 0);
    if (lane == 0) bits[w] = on;
  }
}

__device__ __forceinline__ bool tile_bit(const uint32_t* bits, int t) {
  return (bits[t >> 5] >> (t & 31)) & 1u;
}

// The first t' >= t with bit t' set, or `end` if there is none below end.
__device__ __forceinline__ int next_tile_bit(const uint32_t* bits, int t, int end) {
  while (t < end) {
    const uint32_t w = bits[t >> 5] >> (t & 31);
    if (w) return min(t + __ffs(w) - 1, end);
    t = (t | 31) + 1;
  }
  return end;
}

// ---------------------------------------------------------------------------
// Dropout: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011), from its published definition: ten
// rounds; each multiplies counter words 0 and 2 by M0 = 0xD2511F53 and
// M1 = 0xCD9E8D57 (64-bit products) and maps (c0, c1, c2, c3) to
// (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key
// is bumped by the Weyl constants W0 = 0x9E3779B9, W1 = 0xBB67AE85 between
// rounds.
//
// Element (i, j) of head bh uses the call with counter (j / 8, i, bh, offset);
// its four output words hold eight 16-bit uniforms, key j taking the low
// (j even) or high (j odd) half of word (j % 8) / 2, and the element is kept
// when that uniform is >= t.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)c0 * 0xD2511F53u;  // one wide multiply: both halves
    const uint64_t p1 = (uint64_t)c2 * 0xCD9E8D57u;
    c0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    c1 = (uint32_t)p1;
    c2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    c3 = (uint32_t)p0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Per-halfword keep masks of one output word: 0xFFFF where the uniform >= t.
__device__ __forceinline__ uint32_t keep_halves(uint32_t w, uint32_t t) {
  return __vcmpgeu2(w, t | (t << 16));
}

// The keep bits (bit m: key 8g + m) of one call's eight uniforms.
__device__ __forceinline__ uint32_t keep_bits8(uint4 w, uint32_t t) {
  const uint32_t x01 = __byte_perm(keep_halves(w.x, t), keep_halves(w.y, t), 0x6420);
  const uint32_t x23 = __byte_perm(keep_halves(w.z, t), keep_halves(w.w, t), 0x6420);
  // byte k of x01 / x23 is 0xFF when key k / 4 + k is kept: keep one bit per
  // byte, then add the four bytes into the top byte (no carries: distinct bits)
  const uint32_t lo = ((x01 & 0x08040201u) * 0x01010101u) >> 24;
  const uint32_t hi = ((x23 & 0x80402010u) * 0x01010101u) >> 24;
  return lo | hi;
}

// Keep bits of keys key0 + c, c = 0..31 (bit c), of query row i; key0 is a
// multiple of 8 (the forward and dQ kernels: a query row per thread).
__device__ __forceinline__ uint32_t keep_bits_of_row(const DropParams& d, uint32_t bh, int i,
                                                     int key0) {
  uint32_t bits = 0;
#pragma unroll 2
  for (int g = 0; g < 4; ++g) {  // two calls in flight (four: slower)
    const uint4 w = philox4x32_10((uint32_t)(key0 >> 3) + g, (uint32_t)i, bh, d.offset, d.k0, d.k1);
    bits |= keep_bits8(w, d.t) << (8 * g);
  }
  return bits;
}

// Keep bits of query rows q0 + c, c = 0..31 (bit c), for this lane's key (the
// dK/dV kernel: a key per thread).  The eight lanes of each aligned group of
// eight hold eight consecutive keys (key % 8 == lane % 8), and all 32 lanes
// take part: lane L draws the calls of rows q0 + L + 8r (r = 0..3), which
// cover the group's eight keys, and the lanes swap the bits through shuffles.
__device__ __forceinline__ uint32_t keep_bits_of_key(const DropParams& d, uint32_t bh, int key,
                                                     int q0) {
  const int lane = threadIdx.x & 31, m = key & 7;
  uint32_t mine = 0;  // byte r: the group's keys for row q0 + (lane % 8) + 8r
#pragma unroll
  for (int r = 0; r < 4; ++r) {  // four independent calls in flight
    const uint4 w = philox4x32_10((uint32_t)key >> 3, (uint32_t)(q0 + (lane & 7) + 8 * r), bh,
                                  d.offset, d.k0, d.k1);
    mine |= keep_bits8(w, d.t) << (8 * r);
  }
  uint32_t out = 0;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t k = __shfl_sync(0xffffffffu, mine, (lane & ~7) | s);
    out |= ((k >> m) & 0x01010101u) << s;  // rows s + 8r -> bits s + 8r
  }
  return out;
}

// ---------------------------------------------------------------------------
// Additive score bias: kCount values of keys [k0, k0 + kCount) of one bias
// row, times log2(e) (the kernels work in base 2); 0 past n_keys or without a
// row (brow nullptr: a query row past the end).  The row is 16-byte aligned
// and k0 a multiple of 4, so whole rows are read 4 floats at a time.
// ---------------------------------------------------------------------------
template <int kCount>
__device__ __forceinline__ void load_bias_row(const float* brow, int k0, int n_keys, float* out) {
  constexpr float kL2e = 1.4426950408889634f;
  if (brow && k0 + kCount <= n_keys) {
#pragma unroll
    for (int g = 0; g < kCount / 4; ++g) {
      const float4 t = __ldg(reinterpret_cast<const float4*>(brow + k0) + g);
      out[4 * g] = t.x * kL2e;
      out[4 * g + 1] = t.y * kL2e;
      out[4 * g + 2] = t.z * kL2e;
      out[4 * g + 3] = t.w * kL2e;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kCount; ++e)
      out[e] = (brow && k0 + e < n_keys) ? __ldg(brow + k0 + e) * kL2e : 0.f;
  }
}

// ---------------------------------------------------------------------------
// Grid order: CTA lin -> (work-order index t, head bh) with the heads taken
// `group` at a time, so that the CTAs resident at once share the K / V (or
// Q / dO) tiles of a few heads in L2 instead of all of them; within a group
// the order index runs slowest (t = 0 first: the callers put the heaviest
// tiles there).  A last, smaller group takes the remaining heads.  The host
// picks the group (grid_group_heads): all heads when the inputs fit in L2.
// ---------------------------------------------------------------------------

// Tile taken by order index t: entry t of a block-sparse work order when the
// caller gives one (clamped to [0, n)), else `fallback`.
__device__ __forceinline__ int ordered_tile(const int32_t* order, int t, int n, int fallback) {
  return order ? min(max(__ldg(order + t), 0), n - 1) : fallback;
}

__device__ __forceinline__ void grid_order(int lin, int BH, int nt, int group, int* t, int* bh) {
  const int per_group = group * nt;
  const int g = lin / per_group;
  const int r = lin - g * per_group;
  const int gh = min(group, BH - g * group);  // heads in this group
  *t = r / gh;
  *bh = g * group + (r - *t * gh);
}

// One arrival for the whole warp, made by lane 0 once every lane has got
// here: the lanes' earlier writes (completed TMEM stores, shared-memory
// stores fenced for the async proxy) are ordered before it by the warp sync.
__device__ __forceinline__ void mbar_arrive_warp(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch.  A kernel launched with it (launch_pdl) may
// be resident before the kernel ahead of it on the stream has finished:
// pdl_wait() returns once that kernel has completed and its memory is
// visible, so every kernel calls it before its first global-memory access.
// pdl_launch_dependents() lets the kernel behind it become resident once
// every CTA of this one has called it (or exited); a CTA calls it after its
// TMEM allocation, so that a waiting dependent never holds TMEM columns that
// a CTA of this kernel still has to allocate.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// generic-proxy shared-memory writes -> visible to the async proxy (MMA, TMA)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 / TMEM
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T    (kind::f16: bf16 inputs, fp32 accumulate)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive once on `bar` when every previously issued MMA of this thread is done
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, dense.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A major (0 = K, 1 = MN), 16 B major, 17-22 N>>3, 24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for the 128-byte-swizzled canonical layout
// (8 rows x 128 bytes per 1024-byte swizzle atom, 16-byte chunk index XOR row%8):
//   bits 0-13 start address >> 4, 16-29 leading-dimension byte offset >> 4,
//   32-45 stride-dimension byte offset >> 4, 46-47 version (1),
//   49-51 base offset (0: atoms are 1024-byte aligned), 61-63 layout (2 = SW128).
// K-major operand: rows are M (or N) indices, 64 bf16 of K per 128-byte row;
//   SBO = 1024 (next group of 8 rows), LBO unused; a K step of 16 adds 32 bytes.
// MN-major operand: rows are K indices, 64 bf16 of M/N per 128-byte row;
//   SBO = 1024 (next group of 8 K rows), LBO = byte stride between 64-wide M/N
//   chunks; a K step of 16 adds 2048 bytes.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Byte offset of element (row, col) of a [rows x 64] bf16 block stored in the
// 128-byte-swizzled layout that TMA writes with CU_TENSOR_MAP_SWIZZLE_128B.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col) {
  const uint32_t chunk = (uint32_t)(col >> 3) ^ (uint32_t)(row & 7);
  return (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u + chunk * 16u +
         (uint32_t)(col & 7) * 2u;
}

// TMEM loads/stores, 32 lanes x 32 bits shape: thread t of the warp reads lane
// (lane base + t), N consecutive 32-bit columns.
// A 32-column load with the wait for its completion inside the same asm
// statement, so that no use of the destination registers can be scheduled
// before the wait.
#define FA_TMEM_LD32_SYNC(taddr, r)                                                              \
  asm volatile(                                                                                  \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"   \
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"       \
      "tcgen05.wait::ld.sync.aligned;"                                                           \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),            \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),            \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])             \
      : "r"(taddr)                                                                               \
      : "memory")

// 64-column load with its wait in the same asm statement.
#define FA_TMEM_LD64_SYNC(taddr, r)                                                              \
  asm volatile(                                                                                  \
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"                                     \
      "tcgen05.wait::ld.sync.aligned;"                                                           \
      :                                                                                          \
        "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),                    \
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),                    \
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),                    \
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),                    \
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),                    \
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),                    \
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),                    \
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])                    \
      : "r"(taddr)                                                                               \
      : "memory")

// 16-column load with its wait, and an 8-column store.
#define FA_TMEM_LD16_SYNC(taddr, r)                                                              \
  asm volatile(                                                                                  \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"   \
      "%14,%15}, [%16];\n"                                                                        \
      "tcgen05.wait::ld.sync.aligned;"                                                           \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15])                                                                 \
      : "r"(taddr)                                                                               \
      : "memory")

#define FA_TMEM_ST8(taddr, r)                                                                   \
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"( \
                   taddr),                                                                      \
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),     \
               "r"(r[7]))

#define FA_TMEM_ST16(taddr, r)                                                                  \
  asm volatile(                                                                                 \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"   \
      "%13,%14,%15,%16};" ::"r"(taddr),                                                         \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),   \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),         \
      "r"(r[15]))

#define FA_TMEM_ST32(taddr, r)                                                                   \
  asm volatile(                                                                                  \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"    \
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"( \
          taddr),                                                                                \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),    \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),          \
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),        \
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),        \
      "r"(r[29]), "r"(r[30]), "r"(r[31]))

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32x2 arithmetic (two lanes per instruction).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Maximum of 32 scores held as fp32 bit patterns (four independent chains of
// 3-input maxima), and masking of the keys e >= lim of such a group to -inf.
__device__ __forceinline__ float max32(const uint32_t* r) {
  float mx[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    mx[k] = fmaxf(max3(__uint_as_float(r[8 * k]), __uint_as_float(r[8 * k + 1]),
                       __uint_as_float(r[8 * k + 2])),
                  max3(__uint_as_float(r[8 * k + 3]), max3(__uint_as_float(r[8 * k + 4]),
                                                           __uint_as_float(r[8 * k + 5]),
                                                           __uint_as_float(r[8 * k + 6])),
                       __uint_as_float(r[8 * k + 7])));
  return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

__device__ __forceinline__ void mask32(uint32_t* r, int lim) {  // keys e >= lim are invisible
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (e >= lim) r[e] = 0xff800000u;  // -inf
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace fa
