// Forward pass of exact attention on sm_103a tensor cores: the kernel of d = 64
// calls with dropout or an additive bias (d = 64 without them takes
// fa_fwd64_sm103.cu, and every d = 128 call fa_fwd128s_sm103.cu).
//
// Each query row keeps a running max m, a running denominator l and an
// unnormalised output O that are updated tile by tile over the visible 128-key
// tiles K_j, V_j ("FlashAttention: Fast and Memory-Efficient Exact Attention
// with IO-Awareness", summary page, "Method": block statistics m~, P~, l~
// merged into the running m, l and the rescaled output; blog review "From
// Online Softmax to FlashAttention", "Algorithm FlashAttention (Tiling)").  The
// division by l is deferred to the end, which is the same quantity.
//
// One CTA owns one 128-row query tile (S / P [0, 128), O [128, 192) of 256 TMEM
// columns, 81 KB of shared memory), and two CTAs share an SM: one's set-up,
// first loads and epilogue run under the other's work, and a CTA walks only
// the key tiles its own tile sees.
//
// Roles (192 threads):
//   warps 0-3  softmax: thread t owns row t (TMEM lane t); reads its 128 scores
//              (max, then exponentials), masks, updates m and l, writes
//              P~ = 2^(c S - m) as packed bf16 over the S columns, rescales O
//              in TMEM when m grew by more than 8 in log2 units (lazy
//              rescale), and at the end writes O / l and lse.
//   warp 4     TMA producer: the Q tile once, then K_j / V_j into a ring.
//   warp 5     MMA issuer (one thread).
// Scores are kept in base 2: c = scale * log2(e); lse = ln2 * (m + log2 l).
//
// Every tensor is read through a 4-D TMA descriptor (column, row, head, batch)
// carrying its own strides, and O is stored through its strides, so any layout
// with contiguous rows costs nothing.  A block-sparse CTA copies its row of the
// tile mask into a shared-memory bitmap first.  Dropout: a row's 128 keep bits
// of a tile are drawn before the wait for its scores; dropped entries of P~ are
// zeroed after l has summed them; O is scaled by 1/(1-p) at the end.  The bias
// is added to the scaled scores in the max pass, and the biased scores are
// written back over S.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units: P~ stays below 2^8

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / 64;             // 64-column (128-byte) chunks
  static constexpr int kTileBytes = 128 * D * 2;     // one Q, K or V tile
  static constexpr int kChunkBytes = 128 * 128;      // 128 rows x 128 bytes
  static constexpr int kStages = 2;                  // K/V ring: two CTAs fit an SM
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kSmem = kOffV + kStages * kTileBytes + 1024;  // + alignment slack
  static constexpr int kTmemCols = 256;                              // S, O
  static constexpr int kProducerWarp = 4;  // warps 0-3: softmax
  static constexpr int kIssuerWarp = 5;
  static constexpr int kThreads = 32 * 6;
  static constexpr int kMinBlocks = 2;                               // CTAs per SM
};

struct FwdParams {
  __nv_bfloat16* o;
  Layout lo;
  DropParams drop;
  const float* bias;  // additive score bias or nullptr
  Layout lb;
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

// Key tiles j < jend that the CTA's query tile sees: all of them, or those set
// in its block-mask row (a shared-memory bitmap).
struct KTiles {
  const uint32_t* bits;
  int jend;
  __device__ int next(int j) const { return bits ? next_tile_bit(bits, j, jend) : j; }
};

// Softmax of one query tile for one key tile.  The row max is taken over the
// thread's 128 scores (two 64-column TMEM loads, eight independent 3-input max
// chains); the scores are then reloaded 64 at a time (a TMEM load costs a few
// tens of cycles), exponentiated with packed fp32x2 arithmetic and eight
// independent partial sums, and P~ is written back over the S columns as
// packed bf16.  Boundary tiles (causal diagonal, key padding, the end of the
// sequence) mask invisible keys to -inf.  O is rescaled when the max moved.
// tS / tO include this warp's lane offset.
__device__ __forceinline__ void mask_tail(uint32_t* r, int lim) {  // keys e >= lim are invisible
#pragma unroll
  for (int e = 0; e < 64; ++e)
    if (e >= lim) r[e] = 0xff800000u;  // -inf
}

__device__ __forceinline__ float max64(const uint32_t* r) {
  float mx[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    mx[k] = fmaxf(max3(__uint_as_float(r[8 * k]), __uint_as_float(r[8 * k + 1]),
                       __uint_as_float(r[8 * k + 2])),
                  max3(__uint_as_float(r[8 * k + 3]), max3(__uint_as_float(r[8 * k + 4]),
                                                           __uint_as_float(r[8 * k + 5]),
                                                           __uint_as_float(r[8 * k + 6])),
                       __uint_as_float(r[8 * k + 7])));
  return fmaxf(max3(mx[0], mx[1], mx[2]), max3(mx[3], max3(mx[4], mx[5], mx[6]), mx[7]));
}

// kExtra: the variant with dropout (kbits) and an additive bias (brow: this
// row's bias, nullptr past the end; bias_on warp-uniform).
template <bool kExtra>
__device__ __forceinline__ void softmax_tile(uint32_t tS, uint32_t tO, int ocols32, int key0,
                                             int kv_limit, int row, bool causal, float scale_log2,
                                             bool first, float& m, float& l, uint64_t* p_half,
                                             const uint32_t* kbits, bool bias_on,
                                             const float* brow, int n_keys) {
  // keys [0, lim) of the tile are visible from this row
  int lim = kv_limit - key0;
  if (causal) lim = min(lim, row - key0 + 1);
  const bool partial = lim < 128;
  float tmax;
  float exp_scale = scale_log2;  // multiplies what the exponent pass reads from tS
  if (kExtra && bias_on) {
    // biased scores in log2 units, S scale log2(e)... + bias log2(e), written back
    // over S so that the exponent pass reads them directly
    tmax = -INFINITY;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      uint32_t r[64];
      float bv[64];
      FA_TMEM_LD64_SYNC(tS + 64 * half, r);
      if (partial) mask_tail(r, lim - 64 * half);
      load_bias_row<64>(brow, key0 + 64 * half, n_keys, bv);
#pragma unroll
      for (int e = 0; e < 64; ++e)
        r[e] = __float_as_uint(fmaf(__uint_as_float(r[e]), scale_log2, bv[e]));
      tmax = fmaxf(tmax, max64(r));
      const uint32_t* r_hi = r + 32;
      FA_TMEM_ST32(tS + 64 * half, r);
      FA_TMEM_ST32(tS + 64 * half + 32, r_hi);
    }
    tmem_wait_st();
    exp_scale = 1.f;
  } else {
    uint32_t r[64];
    FA_TMEM_LD64_SYNC(tS, r);
    if (partial) mask_tail(r, lim);
    tmax = max64(r);
    FA_TMEM_LD64_SYNC(tS + 64, r);
    if (partial) mask_tail(r, lim - 64);
    tmax = fmaxf(tmax, max64(r));
    tmax *= scale_log2;
  }
  const float m_tile = tmax;
  const float m_new = fmaxf(m, m_tile);
  const bool grow = m_new > m + kRescaleThreshold;  // true when m = -inf, m_new finite
  float alpha = 1.f;
  if (grow) {
    alpha = (m == -INFINITY) ? 0.f : ex2(m - m_new);
    m = m_new;
  }
  // O holds the sum up to the previous key tile (its P V is complete: this
  // tile's S was issued after it); rescale when the running max moved -- before
  // any of this tile's P is released to the tensor core
  if (!first && __any_sync(0xffffffffu, grow)) {
    for (int c = 0; c < ocols32; ++c) {
      uint32_t o[32];
      FA_TMEM_LD32_SYNC(tO + c * 32, o);
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
      FA_TMEM_ST32(tO + c * 32, o);
    }
  }
  const float nm = (m == -INFINITY) ? 0.f : -m;
  const float2 c2 = make_float2(exp_scale, exp_scale), nm2 = make_float2(nm, nm);
  float2 acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = make_float2(0.f, 0.f);
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint32_t r[64];
    FA_TMEM_LD64_SYNC(tS + 64 * half, r);
    if (partial) mask_tail(r, lim - 64 * half);
    uint32_t pk[32];
    // dropout: keep bits of this half's keys [0, 32) and [32, 64)
    const uint32_t kb0 = kExtra ? (half ? kbits[2] : kbits[0]) : 0u;
    const uint32_t kb1 = kExtra ? (half ? kbits[3] : kbits[1]) : 0u;
#pragma unroll
    for (int e = 0; e < 64; e += 2) {
      const float2 xx = fma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), c2, nm2);
      float2 pv = make_float2(ex2(xx.x), ex2(xx.y));
      acc[(e >> 1) & 7] = add2(acc[(e >> 1) & 7], pv);  // l sums the undropped P~
      if constexpr (kExtra) {  // dropout (all bits set without it)
        const uint32_t kb = e < 32 ? kb0 : kb1;
        if (!((kb >> (e & 31)) & 1u)) pv.x = 0.f;
        if (!((kb >> ((e + 1) & 31)) & 1u)) pv.y = 0.f;
      }
      pk[e >> 1] = pack_bf16(pv.x, pv.y);
    }
    // packed P of keys [64 half, 64 half + 64) over S columns [32 half, 32 half + 32),
    // which this thread has already read
    FA_TMEM_ST32(tS + 32 * half, pk);
    if (half == 0) {
      // keys [0, 64) of P are in place (and O rescaled): the first half of
      // O += P V may start while the second half of P is computed
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(p_half);
    }
  }
  const float2 s01 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
  const float2 s23 = add2(add2(acc[4], acc[5]), add2(acc[6], acc[7]));
  const float2 st = add2(s01, s23);
  l = l * alpha + (st.x + st.y);
  tmem_wait_st();
}

template <int D, bool kExtra>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, FwdCfg<D>::kMinBlocks)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t q_full, drain, s_full, p_half, p_full, o_done;
  __shared__ uint64_t k_full[C::kStages], v_full[C::kStages], k_empty[C::kStages],
      v_empty[C::kStages];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ uint32_t mask_bits[kMaskBitmapWords];  // block-mask row qi

  pdl_wait();  // the kernel ahead on the stream is done (it may write our inputs)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heaviest query tiles first: causal rows near the end see the most keys; a
  // block-sparse work order lists the query tiles by their visible key tiles
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
    mbar_init(&drain, 1);
    mbar_init(&s_full, 1);
    mbar_init(&p_half, 4);  // one arrival per softmax warp: keys [0, 64) of P
    mbar_init(&p_full, 4);  // all of P
    mbar_init(&o_done, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kIssuerWarp) tmem_alloc(&tmem_slot, C::kTmemCols);
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
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_4d(&tmQ, &q_full, smem + C::kOffQ + c * C::kChunkBytes, c * 64, qi * 128, hd, b);
      int kcount[C::kStages] = {}, vcount[C::kStages] = {};
      int u = 0;
      bool ok = true;
      for (int j = jfirst; j < tiles.jend && ok; j = tiles.next(j + 1), ++u) {
        const int st = u % C::kStages;
        const uint32_t ph = (u / C::kStages) & 1;
        ok = mbar_wait(&k_empty[st], ph ^ 1, &abort_flag, p.status, 101);
        if (!ok) break;
        mbar_expect_tx(&k_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(&tmK, &k_full[st], smem + C::kOffK + st * C::kTileBytes + c * C::kChunkBytes,
                      c * 64, j * 128, hd, b);
        ++kcount[st];
        ok = mbar_wait(&v_empty[st], ph ^ 1, &abort_flag, p.status, 102);
        if (!ok) break;
        mbar_expect_tx(&v_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(&tmV, &v_full[st], smem + C::kOffV + st * C::kTileBytes + c * C::kChunkBytes,
                      c * 64, j * 128, hd, b);
        ++vcount[st];
      }
      // every issued copy must have landed before the CTA may exit
      mbar_drain(&q_full, 0);
      for (int s = 0; s < C::kStages; ++s) {
        if (kcount[s]) mbar_drain(&k_full[s], (kcount[s] - 1) & 1);
        if (vcount[s]) mbar_drain(&v_full[s], (vcount[s] - 1) & 1);
      }
    }
  } else if (warp == C::kIssuerWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
      const uint64_t dQ = sdesc_sw128(smem_addr(smem + C::kOffQ), 16, 1024);
      const uint32_t sK = smem_addr(smem + C::kOffK);
      const uint32_t sV = smem_addr(smem + C::kOffV);
      const uint32_t tS = tmem, tO = tmem + 128;
      bool ok = mbar_wait(&q_full, 0, &abort_flag, p.status, 201);
      int u = 0;
      for (int j = jfirst; ok && j < tiles.jend; j = tiles.next(j + 1), ++u) {
        const int st = u % C::kStages;
        const uint32_t ph = (u / C::kStages) & 1;
        ok = mbar_wait(&k_full[st], ph, &abort_flag, p.status, 202);
        // S = Q K_j^T, after the previous P V (its P sits in the S columns)
        if (ok && u > 0) ok = mbar_wait(&o_done, (u - 1) & 1, &abort_flag, p.status, 203);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dK = sdesc_sw128(sK + st * C::kTileBytes, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * C::kChunkBytes + (ks & 3) * 32) >> 4;
          mma_ss(tS, dQ + off, dK + off, idesc_qk, ks > 0 ? 1u : 0u);
        }
        mma_commit(&s_full);
        mma_commit(&k_empty[st]);
        ok = mbar_wait(&v_full[st], ph, &abort_flag, p.status, 207);
        if (!ok) break;
        // O += P V_j, P read from TMEM (packed, 8 columns per 16 keys): keys
        // [0, 64) as soon as the softmax has written them, then the rest
        const uint64_t dV = sdesc_sw128(sV + st * C::kTileBytes, C::kChunkBytes, 1024);
        ok = mbar_wait(&p_half, u & 1, &abort_flag, p.status, 209);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ts(tO, tS + ks * 8, dV + ks * (2048 >> 4), idesc_pv, (u > 0 || ks > 0) ? 1u : 0u);
        ok = mbar_wait(&p_full, u & 1, &abort_flag, p.status, 205);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 4; ks < 8; ++ks)
          mma_ts(tO, tS + ks * 8, dV + ks * (2048 >> 4), idesc_pv, 1u);
        mma_commit(&o_done);
        mma_commit(&v_empty[st]);
      }
      // all MMAs issued by this thread are complete once its drain flips
      mma_commit(&drain);
      mbar_drain(&drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int row = qi * 128 + (tid & 127);
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off, tO = tmem + 128 + lane_off;
    float m = -INFINITY, l = 0.f;
    int n = 0;
    bool ok = true;
    // additive bias: this row's [N] bias (nullptr past the end of the sequence)
    const bool bias_on = kExtra && p.bias != nullptr;
    const float* brow = (bias_on && row < p.N) ? p.bias + row_offset(p.lb, b, hd, row) : nullptr;
    for (int j = jfirst; j < tiles.jend; j = tiles.next(j + 1), ++n) {
      // dropout: this row's keep bits of the tile, drawn before S is waited for
      uint32_t kbits[4] = {~0u, ~0u, ~0u, ~0u};
      if constexpr (kExtra) {
        if (p.drop.t) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            kbits[c] = keep_bits_of_row(p.drop, (uint32_t)bh, row, j * 128 + 32 * c);
        }
      }
      ok = mbar_wait_warp(&s_full, n & 1, &abort_flag, p.status, 301);
      if (!ok) break;
      tc_fence_after();
      softmax_tile<kExtra>(tS, tO, D / 32, j * 128, kv_limit, row, p.causal != 0, p.scale_log2,
                           n == 0, m, l, &p_half, kbits, bias_on, brow, p.N);
      tc_fence_before();
      mbar_arrive_warp(&p_full);
    }
    // ------------------------------------------------------------ epilogue
    if (ok) {
      bool have = n > 0;
      if (have) {
        have = mbar_wait_warp(&o_done, (n - 1) & 1, &abort_flag, p.status, 304);
        tc_fence_after();
      }
      if (__all_sync(0xffffffffu, !abort_flag)) {  // warp-uniform: TMEM loads below
        const bool empty_row = !(l > 0.f);
        // dropout: the kept entries of P are scaled by 1 / (1 - p)
        const float inv = empty_row ? 0.f : (kExtra ? p.drop.rp : 1.f) / l;
        const long long base = row_offset(p.lo, b, hd, row);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          if (have) {
            FA_TMEM_LD32_SYNC(tO + c * 32, r);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = 0u;
          }
          if (row < p.N) {
            uint4* dst = reinterpret_cast<uint4*>(p.o + base + c * 32);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const float* f = reinterpret_cast<const float*>(r + g * 8);
              uint4 w;
              w.x = pack_bf16(f[0] * inv, f[1] * inv);
              w.y = pack_bf16(f[2] * inv, f[3] * inv);
              w.z = pack_bf16(f[4] * inv, f[5] * inv);
              w.w = pack_bf16(f[6] * inv, f[7] * inv);
              dst[g] = w;
            }
          }
        }
        if (row < p.N)
          p.lse[(size_t)bh * p.N + row] = empty_row ? -INFINITY : (m + __log2f(l)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kIssuerWarp) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t s) {
  using C = FwdCfg<D>;
  const int BH = a.B * a.H;
  CUtensorMap mq, mk, mv;
  if (!encode_bhnd_map(&mq, a.q, a.lq, a.B, a.H, a.N, D, 128) ||
      !encode_bhnd_map(&mk, a.k, a.lk, a.B, a.H, a.N, D, 128) ||
      !encode_bhnd_map(&mv, a.v, a.lv, a.B, a.H, a.N, D, 128))
    return cudaErrorInvalidValue;
  FwdParams p;
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
  p.drop = a.drop;
  p.bias = a.bias;
  p.lb = a.lb;
  // calls without dropout or a bias take fa_fwd64_sm103.cu: only the variant
  // with them is launched here
  auto kernel = fa_fwd_kernel<D, true>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(p.T * BH), dim3(C::kThreads), C::kSmem, s, mq, mk, mv, p);
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t s) {
  if (a.d == 128) return launch_fwd128s_bf16(a, s);
  if (!a.drop.t && !a.bias) return launch_fwd64_bf16(a, s);
  return launch_fwd_d<64>(a, s);
}

}  // namespace fa
