// Forward pass of exact attention at d = 64 on sm_103a tensor cores, with each
// key tile's softmax split between two warpgroups ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", summary page, "Method":
// the softmax of a row is assembled from blocks, each with its own statistics
// m, l, and the partial results are merged by rescaling them to the common
// maximum; blog review, "Algorithm FlashAttention (Tiling)").
//
// One CTA owns a 128-row query tile of one (batch, head); two CTAs share an SM.
// Warpgroup h (h = 0, 1) owns keys [64h, 64h+64) of every key tile and keeps
// its own running statistics m_h, l_h and its own output accumulator O_h:
//   S_h   = Q K_h^T            (N = 64)      into TMEM columns [64h, 64h+64)
//   P~_h  = 2^(c S_h - m_h)    packed bf16 over columns [64h, 64h+32)
//   O_h   = O_h 2^(m_old - m_h) (lazily, when m_h grows by more than 8) + P~_h V_h
// so each thread exponentiates 64 scores per key tile instead of 128, and the
// two halves form independent chains S_h -> P~_h -> P~_h V_h -> next S_h, each
// with its own MMA-issuing thread.  At the end the two warpgroups exchange
// (m_h, l_h) through shared memory and write
//   O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / l,  l = l_0 2^(m_0 - m) + l_1 2^(m_1 - m),
//   m = max(m_0, m_1),  lse = ln2 (m + log2 l).
// TMEM (256 columns): S [0,128), O_0 [128,192), O_1 [192,256).
// Roles (352 threads): warps 0-3 softmax of keys [0,64), warps 4-7 of keys
// [64,128) (thread = query row), warp 8 TMA producer (Q once; K/V ring of 2),
// warps 9, 10 MMA issuers for halves 0, 1 (one thread each).
// This is the kernel of d = 64 calls without dropout or a bias.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units: P~ stays below 2^8

struct Fwd64Cfg {
  static constexpr int D = 64;
  static constexpr int kTileBytes = 128 * D * 2;  // one Q, K or V tile (one 128-byte-row chunk)
  static constexpr int kStages = 2;               // K/V ring
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kSmem = kOffV + kStages * kTileBytes + 1024;  // + alignment slack
  static constexpr int kTmemCols = 256;
  static constexpr uint32_t kColS = 0, kColO = 128;  // S_h at 64 h, O_h at kColO + 64 h
  static constexpr int kSoftmaxWarps = 8;
  static constexpr int kProducerWarp = 8;
  static constexpr int kIssuerWarp0 = 9;
  static constexpr int kThreads = 32 * 11;
};

struct Fwd64Params {
  __nv_bfloat16* o;
  Layout lo;
  float* lse;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  const int32_t* order;  // block-sparse work order (query tiles) or nullptr
  int H, N, T, BH;
  int group;  // heads per group of the grid order
  float scale_log2;
  int causal;
  int* status;
};

// Key tiles j that query tile qi sees: j < jend (causal diagonal, key
// padding, end of sequence), block-mask row qi (as a shared-memory bitmap;
// nullptr: no block mask).
struct KTiles {
  const uint32_t* bits;
  int jend;
  __device__ int next(int j) const { return bits ? next_tile_bit(bits, j, jend) : j; }
};

// Softmax of this warpgroup's 64 keys of one key tile for this thread's row:
// keys [0, lim) visible.  tS: the half's S columns, tO: its O columns (lane
// offset included).
__device__ __forceinline__ void softmax_half(uint32_t tS, uint32_t tO, int lim, float scale_log2,
                                             bool first, float& m, float& l) {
  float tmax;
  {
    uint32_t r[32];
    FA_TMEM_LD32_SYNC(tS, r);
    if (lim < 32) mask32(r, lim);
    tmax = max32(r);
    FA_TMEM_LD32_SYNC(tS + 32, r);
    if (lim < 64) mask32(r, lim - 32);
    tmax = fmaxf(tmax, max32(r)) * scale_log2;
  }
  const float m_new = fmaxf(m, tmax);
  const bool grow = m_new > m + kRescaleThreshold;  // true when m = -inf, m_new finite
  float alpha = 1.f;
  if (grow) {
    alpha = (m == -INFINITY) ? 0.f : ex2(m - m_new);
    m = m_new;
  }
  // O_h holds the sum up to the previous key tile (its P V is complete: this
  // tile's S was issued after it); rescale when the running max moved, before
  // this tile's P is released to the tensor core
  if (!first && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      uint32_t o[32];
      FA_TMEM_LD32_SYNC(tO + 32 * c, o);
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
      FA_TMEM_ST32(tO + 32 * c, o);
    }
  }
  const float nm = (m == -INFINITY) ? 0.f : -m;
  const float2 c2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(nm, nm);
  float2 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float2(0.f, 0.f);
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    uint32_t r[32];
    FA_TMEM_LD32_SYNC(tS + 32 * c, r);
    if (lim < 64) mask32(r, lim - 32 * c);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const float2 xx = fma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), c2, nm2);
      const float2 pv = make_float2(ex2(xx.x), ex2(xx.y));
      acc[(e >> 1) & 3] = add2(acc[(e >> 1) & 3], pv);
      pk[e >> 1] = pack_bf16(pv.x, pv.y);
    }
    // packed P of keys [32c, 32c + 32) over S columns [16c, 16c + 16), which
    // this thread has already read
    FA_TMEM_ST16(tS + 16 * c, pk);
  }
  const float2 st = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
  l = l * alpha + (st.x + st.y);
  tmem_wait_st();
}

__global__ void __launch_bounds__(Fwd64Cfg::kThreads, 2)
    fa_fwd64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Fwd64Params p) {
  using C = Fwd64Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t q_full, drain[2];
  // per half h: s_full (S_h in TMEM), p_full (P~_h written, one arrival per
  // warp of warpgroup h), o_done (P~_h V_h done: the S_h columns are free and
  // O_h is current).  Per stage: k_empty / v_empty count one commit from each
  // issuer.  Each next phase of a barrier needs its waiter's own progress
  // first, so no waiter falls a phase behind.
  __shared__ uint64_t s_full[2], p_full[2], o_done[2];
  __shared__ uint64_t k_full[C::kStages], v_full[C::kStages], k_empty[C::kStages],
      v_empty[C::kStages];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float s_m[2][128], s_l[2][128];  // each half's final statistics, by row
  __shared__ uint32_t mask_bits[kMaskBitmapWords];  // block-mask row qi

  pdl_wait();  // the kernel ahead on the stream is done (it may write our inputs)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // causal: the last query tiles see the most keys: first; a block-sparse work
  // order lists the query tiles by their visible key tiles
  int order, bh;
  grid_order(blockIdx.x, p.BH, p.T, p.group, &order, &bh);
  const int qi = ordered_tile(p.order, order, p.T, p.T - 1 - order);
  const int b = bh / p.H;
  const int hd = bh - b * p.H;
  int kv_limit = p.N;
  if (p.kv_len) kv_limit = max(0, min(p.kv_len[b], p.N));
  const int jkv = (kv_limit + 127) / 128;
  if (p.block_mask) build_tile_bitmap(mask_bits, p.block_mask + (size_t)qi * p.T, 1, p.T);
  const KTiles tiles{p.block_mask ? mask_bits : nullptr, p.causal ? min(jkv, qi + 1) : jkv};

  if (tid == 0) {
    mbar_init(&q_full, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&drain[h], 1);
      mbar_init(&s_full[h], 1);
      mbar_init(&p_full[h], 4);
      mbar_init(&o_done[h], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 2);
      mbar_init(&v_empty[s], 2);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kIssuerWarp0) tmem_alloc(&tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  pdl_launch_dependents();  // TMEM held: the next kernel may become resident
  const int jfirst = tiles.next(0);  // after the barrier: the bitmap is complete

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      mbar_expect_tx(&q_full, C::kTileBytes);
      tma_load_4d(&tmQ, &q_full, smem + C::kOffQ, 0, qi * 128, hd, b);
      int kcount[C::kStages] = {}, vcount[C::kStages] = {};
      int u = 0;
      bool ok = true;
      for (int j = jfirst; j < tiles.jend && ok; j = tiles.next(j + 1), ++u) {
        const int st = u % C::kStages;
        const uint32_t ph = (u / C::kStages) & 1;
        ok = mbar_wait(&k_empty[st], ph ^ 1, &abort_flag, p.status, 2301);
        if (!ok) break;
        mbar_expect_tx(&k_full[st], C::kTileBytes);
        tma_load_4d(&tmK, &k_full[st], smem + C::kOffK + st * C::kTileBytes, 0, j * 128, hd, b);
        ++kcount[st];
        ok = mbar_wait(&v_empty[st], ph ^ 1, &abort_flag, p.status, 2302);
        if (!ok) break;
        mbar_expect_tx(&v_full[st], C::kTileBytes);
        tma_load_4d(&tmV, &v_full[st], smem + C::kOffV + st * C::kTileBytes, 0, j * 128, hd, b);
        ++vcount[st];
      }
      // every issued copy must have landed before the CTA may exit
      mbar_drain(&q_full, 0);
      for (int s = 0; s < C::kStages; ++s) {
        if (kcount[s]) mbar_drain(&k_full[s], (kcount[s] - 1) & 1);
        if (vcount[s]) mbar_drain(&v_full[s], (vcount[s] - 1) & 1);
      }
    }
  } else if (warp >= C::kIssuerWarp0) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer h serves half h: S_h once P~_h of the previous key tile has been
    // read by its P V (o_done), then P~_h V_h once the softmax has written P~_h.
    // Both walk every visible key tile and release each K / V stage with a
    // commit of their own.
    const int h = warp - C::kIssuerWarp0;
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 64, false, false);   // S_h: N = 64 keys
      constexpr uint32_t idesc_pv = idesc_bf16(128, 64, false, true);   // P V: N = d = 64
      const uint64_t dQ = sdesc_sw128(smem_addr(smem + C::kOffQ), 16, 1024);
      const uint32_t sK = smem_addr(smem + C::kOffK), sV = smem_addr(smem + C::kOffV);
      const uint32_t tS = tmem + C::kColS + 64 * h, tO = tmem + C::kColO + 64 * h;
      bool ok = mbar_wait(&q_full, 0, &abort_flag, p.status, 2311);
      int u = 0;
      for (int j = jfirst; ok && j < tiles.jend; j = tiles.next(j + 1), ++u) {
        const int st = u % C::kStages;
        const uint32_t ph = (u / C::kStages) & 1;
        ok = mbar_wait(&k_full[st], ph, &abort_flag, p.status, 2312);
        if (ok && u > 0) ok = mbar_wait(&o_done[h], (u - 1) & 1, &abort_flag, p.status, 2313 + h);
        if (!ok) break;
        tc_fence_after();
        // keys [64h, 64h + 64) of the tile: 64 rows x 128 bytes into it
        const uint64_t dK = sdesc_sw128(sK + st * C::kTileBytes + 64 * 128 * h, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tS, dQ + ((kk * 32) >> 4), dK + ((kk * 32) >> 4), idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(&s_full[h]);
        mma_commit(&k_empty[st]);
        ok = mbar_wait(&v_full[st], ph, &abort_flag, p.status, 2315);
        if (ok) ok = mbar_wait(&p_full[h], u & 1, &abort_flag, p.status, 2316 + h);
        if (!ok) break;
        tc_fence_after();
        // O_h += P~_h V_h: P~ of 16 keys per 8 packed columns; V rows 64h + 16kk
        // (d contiguous: MN-major)
        const uint64_t dV = sdesc_sw128(sV + st * C::kTileBytes + 64 * 128 * h, 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(tO, tS + 8 * kk, dV + kk * (2048 >> 4), idesc_pv, (u > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&o_done[h]);
        mma_commit(&v_empty[st]);
      }
      // all MMAs issued by this thread are complete once its drain flips
      mma_commit(&drain[h]);
      mbar_drain(&drain[h], 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int h = warp >> 2;  // key half
    const int tq = tid & 127;
    const int row = qi * 128 + tq;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + C::kColS + 64 * h + lane_off;
    const uint32_t tO = tmem + C::kColO + 64 * h + lane_off;
    float m = -INFINITY, l = 0.f;
    int n = 0;
    bool ok = true;
    for (int j = jfirst; j < tiles.jend; j = tiles.next(j + 1), ++n) {
      ok = mbar_wait_warp(&s_full[h], n & 1, &abort_flag, p.status, 2321 + h);
      if (!ok) break;
      tc_fence_after();
      // keys [key0, key0 + lim) of the half are visible from this row
      const int key0 = j * 128 + 64 * h;
      int lim = kv_limit - key0;
      if (p.causal) lim = min(lim, row - key0 + 1);
      softmax_half(tS, tO, lim, p.scale_log2, n == 0, m, l);
      tc_fence_before();
      mbar_arrive_warp(&p_full[h]);
    }
    // ------------------------------------------------------------ epilogue
    // both halves' accumulators must be complete before either is read
    bool have = ok && n > 0;
    if (have) have = mbar_wait_warp(&o_done[0], (n - 1) & 1, &abort_flag, p.status, 2323);
    if (have) have = mbar_wait_warp(&o_done[1], (n - 1) & 1, &abort_flag, p.status, 2324);
    tc_fence_after();
    s_m[h][tq] = m;
    s_l[h][tq] = l;
    asm volatile("bar.sync 1, 256;" ::: "memory");  // the eight softmax warps
    if (__all_sync(0xffffffffu, !abort_flag)) {  // warp-uniform: TMEM loads below
      const float m0 = s_m[0][tq], m1 = s_m[1][tq];
      const float mm = fmaxf(m0, m1);
      const float a0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - mm);
      const float a1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - mm);
      const float lt = s_l[0][tq] * a0 + s_l[1][tq] * a1;
      const bool empty_row = !(lt > 0.f);
      const float inv = empty_row ? 0.f : 1.f / lt;
      // warpgroup h writes d columns [32h, 32h + 32) of the row
      uint32_t r0[32], r1[32];
      if (have) {
        FA_TMEM_LD32_SYNC(tmem + C::kColO + 32 * h + lane_off, r0);
        FA_TMEM_LD32_SYNC(tmem + C::kColO + 64 + 32 * h + lane_off, r1);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) r0[e] = r1[e] = 0u;
      }
      const float w0 = a0 * inv, w1 = a1 * inv;
      if (row < p.N) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + row_offset(p.lo, b, hd, row) + 32 * h);
        auto f = [&](int e) {
          return __uint_as_float(r0[e]) * w0 + __uint_as_float(r1[e]) * w1;
        };
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 w;
          w.x = pack_bf16(f(8 * g), f(8 * g + 1));
          w.y = pack_bf16(f(8 * g + 2), f(8 * g + 3));
          w.z = pack_bf16(f(8 * g + 4), f(8 * g + 5));
          w.w = pack_bf16(f(8 * g + 6), f(8 * g + 7));
          dst[g] = w;
        }
        if (h == 0)
          p.lse[(size_t)bh * p.N + row] = empty_row ? -INFINITY : (mm + __log2f(lt)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kIssuerWarp0) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace

cudaError_t launch_fwd64_bf16(const FwdArgs& a, cudaStream_t s) {
  using C = Fwd64Cfg;
  const int BH = a.B * a.H;
  CUtensorMap mq, mk, mv;
  if (!encode_bhnd_map(&mq, a.q, a.lq, a.B, a.H, a.N, C::D, 128) ||
      !encode_bhnd_map(&mk, a.k, a.lk, a.B, a.H, a.N, C::D, 128) ||
      !encode_bhnd_map(&mv, a.v, a.lv, a.B, a.H, a.N, C::D, 128))
    return cudaErrorInvalidValue;
  Fwd64Params p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lo = a.lo;
  p.lse = a.lse;
  p.kv_len = a.mask_kind == FA_MASK_KEY_PADDING ? a.kv_len : nullptr;
  p.block_mask = a.mask_kind == FA_MASK_BLOCK_SPARSE ? a.block_mask : nullptr;
  p.H = a.H;
  p.N = a.N;
  p.T = tiles_of(a.N, 128);
  p.order = p.block_mask ? a.tile_order : nullptr;  // query tiles at [0, T)
  p.BH = BH;
  p.group = grid_group_heads(a.B, a.H, a.N, a.d, a.causal);
  p.scale_log2 = a.scale * kLog2e;
  p.causal = a.causal;
  p.status = a.status;
  cudaError_t e =
      cudaFuncSetAttribute(fa_fwd64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(fa_fwd64_kernel, dim3(p.T * BH), dim3(C::kThreads), C::kSmem, s, mq, mk, mv, p);
}

}  // namespace fa
