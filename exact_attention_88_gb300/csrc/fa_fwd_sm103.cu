// Forward pass of exact attention on sm_103a tensor cores.
//
// Each query row keeps a running max m, a running denominator l and an
// unnormalised output O that are updated tile by tile over the visible 128-key
// tiles K_j, V_j ("FlashAttention: Fast and Memory-Efficient Exact Attention
// with IO-Awareness", summary page, "Method": block statistics m~, P~, l~
// merged into the running m, l and the rescaled output; blog review "From
// Online Softmax to FlashAttention", "Algorithm FlashAttention (Tiling)").  The
// division by l is deferred to the end, which is the same quantity.
//
// d = 128 with a block mask (calls without one take fa_fwd128s_sm103.cu, one
// query tile per CTA with two score buffers): one CTA owns two 128-row query tiles (A and B) of one (batch,
// head) and streams the key/value tiles through a shared ring.  The two tiles
// alternate on the tensor core: while one tile's softmax runs on its
// warpgroup, the other tile's S = Q K^T or O += P V is computed, so the tensor
// core has work queued.  TMEM columns: S_A / P_A [0,128), O_A [128, 128+d),
// S_B / P_B [256, 384), O_B [384, 384+d).
// d = 64: one CTA owns one query tile (S / P [0, 128), O [128, 192) of 256
// TMEM columns, 81 KB of shared memory), and two CTAs share an SM: one's
// set-up, first loads and epilogue run under the other's work, and a CTA walks
// only the key tiles its own tile sees.
//
// Roles (d = 128: 352 threads; d = 64: 192):
//   warps 0-3 (, 4-7) softmax of tile A (, B): thread t owns row t (TMEM lane
//                   t); at d = 128 the two take turns key tile by key tile;
//                   reads its 128 scores (max, then exponentials), masks,
//                   updates m and l, writes P~ = 2^(c S - m) as packed bf16
//                   over the S columns,
//                   rescales O in TMEM when m grew by more than 8 in log2 units
//                   (lazy rescale), and at the end writes O / l and lse.
//   warp 8 (4)      TMA producer: the Q tiles once, then K_j / V_j into rings.
//   warps 9, 10 (5) MMA issuers for tile A, B (one thread each).
// Scores are kept in base 2: c = scale * log2(e); lse = ln2 * (m + log2 l).
//
// Every tensor is read through a 4-D TMA descriptor (column, row, head, batch)
// carrying its own strides, and O is stored through its strides, so any layout
// with contiguous rows costs nothing.  A block-sparse CTA copies its rows of
// the tile mask into shared-memory bitmaps first.  The kExtra variant adds
// dropout (a row's 128 keep bits of a tile are drawn before its turn; dropped
// entries of P~ are zeroed after l has summed them; O is scaled by 1/(1-p) at
// the end) and an additive bias (added to the scaled scores in the max pass,
// the biased scores written back over S).
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units: P~ stays below 2^8

template <int D, int kTiles>
struct FwdCfg {
  static constexpr int kChunks = D / 64;             // 64-column (128-byte) chunks
  static constexpr int kTileBytes = 128 * D * 2;     // one Q, K or V tile
  static constexpr int kChunkBytes = 128 * 128;      // 128 rows x 128 bytes
  // K/V ring depth; a one-tile CTA keeps two stages so that two CTAs fit an SM
  static constexpr int kStages = kTiles == 1 ? 2 : (D == 64) ? 3 : 2;
  static constexpr int kOffQ = 0;                    // Q_A (, Q_B)
  static constexpr int kOffK = kOffQ + kTiles * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kSmem = kOffV + kStages * kTileBytes + 1024;  // + alignment slack
  static constexpr int kTmemCols = kTiles == 2 ? 512 : 256;          // (S, O) per tile
  static constexpr int kSoftmaxWarps = 4 * kTiles;
  static constexpr int kProducerWarp = kSoftmaxWarps;
  static constexpr int kIssuerWarp0 = kSoftmaxWarps + 1;             // one issuer per tile
  static constexpr int kThreads = 32 * (kSoftmaxWarps + 1 + kTiles);
  static constexpr int kMinBlocks = kTiles == 2 ? 1 : 2;             // CTAs per SM
  // d = 128 (two tiles): the two softmax warpgroups take turns key tile by key
  // tile, so that each runs alone while the tensor core works for the other
  // tile (run side by side, the two tiles' MMAs bunch up and the pipe idles
  // while both passes run).  d = 64 keeps one query tile per CTA and two CTAs
  // per SM, whose softmax passes run side by side.
  static constexpr bool kTurns = D == 128;
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
  const int32_t* order;  // block-sparse work order of the units (pairs or tiles), or nullptr
  int H, N, T, BH, pairs;
  int group;  // heads per group of the grid order
  float scale_log2;
  int causal;
  int* status;
};

// Visibility of key tile j for the CTA's two query tiles.
struct PairTiles {
  const uint32_t* bits_a;  // block-mask rows as shared-memory bitmaps (nullptr: no block mask)
  const uint32_t* bits_b;
  int jend_a, jend_b;      // tiles j >= jend are invisible (causal / key padding / past N)
  __device__ bool vis_a(int j) const { return j < jend_a && (!bits_a || tile_bit(bits_a, j)); }
  __device__ bool vis_b(int j) const { return j < jend_b && (!bits_b || tile_bit(bits_b, j)); }
  __device__ int next(int j) const {  // next key tile visible to either tile, or end()
    if (!bits_a) return j;            // no block mask: every j < end() is visible to one
    const int na = next_tile_bit(bits_a, j, jend_a);
    const int nb = bits_b ? next_tile_bit(bits_b, j, jend_b) : jend_b;
    const int ea = na < jend_a ? na : end(), eb = nb < jend_b ? nb : end();
    return min(ea, eb);
  }
  __device__ int end() const { return max(jend_a, jend_b); }
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

template <int D, bool kExtra, int kTiles>
__global__ void __launch_bounds__(FwdCfg<D, kTiles>::kThreads, FwdCfg<D, kTiles>::kMinBlocks)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D, kTiles>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t q_full, drain[2];
  __shared__ uint64_t s_full[2], p_half[2], p_full[2], o_done[2], turn[2];  // per query tile
  // turn[x]: tile x's softmax may run.  The two softmax warpgroups take turns
  // key tile by key tile (A, B, A, B, ...), so that each runs alone on the
  // SMSPs while the tensor core works for the other tile.
  __shared__ uint64_t k_full[C::kStages], v_full[C::kStages], k_empty[C::kStages],
      v_empty[C::kStages];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ uint32_t mask_bits[2][kMaskBitmapWords];  // block-mask rows qa, qb

  pdl_wait();  // the kernel ahead on the stream is done (it may write our inputs)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heaviest pairs first: causal rows near the end see the most keys; a
  // block-sparse work order lists the units by their visible tiles
  int order, bh;
  grid_order(blockIdx.x, p.BH, p.pairs, p.group, &order, &bh);
  const int pair = ordered_tile(p.order, order, p.pairs, p.pairs - 1 - order);
  const int b = bh / p.H;
  const int hd = bh - b * p.H;
  // query tiles (p.pairs counts the CTAs' units: pairs of tiles, or tiles)
  const int qa = kTiles == 2 ? 2 * pair : pair, qb = 2 * pair + 1;  // qb may be past the end
  const bool has_b = kTiles == 2 && qb < p.T;

  int kv_limit = p.N;
  if (p.kv_len) kv_limit = max(0, min(p.kv_len[b], p.N));
  const int jkv = (kv_limit + 127) / 128;
  PairTiles tiles;
  tiles.bits_a = p.block_mask ? mask_bits[0] : nullptr;
  tiles.bits_b = (p.block_mask && has_b) ? mask_bits[1] : nullptr;
  if (p.block_mask) {
    build_tile_bitmap(mask_bits[0], p.block_mask + (size_t)qa * p.T, 1, p.T);
    if (has_b) build_tile_bitmap(mask_bits[1], p.block_mask + (size_t)qb * p.T, 1, p.T);
  }
  tiles.jend_a = p.causal ? min(jkv, qa + 1) : jkv;
  tiles.jend_b = !has_b ? 0 : (p.causal ? min(jkv, qb + 1) : jkv);

  if (tid == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_half[x], 4);  // one arrival per softmax warp: keys [0, 64) of P
      mbar_init(&p_full[x], 4);  // all of P
      mbar_init(&turn[x], 4);
      mbar_init(&o_done[x], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], kTiles);  // one commit from each issuer
      mbar_init(&v_empty[s], kTiles);
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

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      mbar_expect_tx(&q_full, (has_b ? 2 : 1) * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_4d(&tmQ, &q_full, smem + C::kOffQ + c * C::kChunkBytes, c * 64, qa * 128, hd, b);
        if (has_b)
          tma_load_4d(&tmQ, &q_full, smem + C::kOffQ + C::kTileBytes + c * C::kChunkBytes, c * 64,
                      qb * 128, hd, b);
      }
      int kcount[C::kStages] = {}, vcount[C::kStages] = {};
      int u = 0;
      bool ok = true;
      for (int j = tiles.next(0); j < tiles.end() && ok; j = tiles.next(j + 1), ++u) {
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
  } else if (warp >= C::kIssuerWarp0) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per query tile (warp 9: A, warp 10: B): an MMA costs
    // its issuing thread about as long as the tensor core takes to run it, so
    // a single thread waiting on one tile's softmax would starve the other
    // tile's MMAs.  Both walk the key tiles either tile sees and release each
    // K / V stage with a commit of their own (the stage barriers count two).
    // (B runs even without a tile B: it still owes its commit for every stage)
    const int x = warp - C::kIssuerWarp0;
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
      const uint64_t dQx = sdesc_sw128(smem_addr(smem + C::kOffQ + x * C::kTileBytes), 16, 1024);
      const uint32_t sK = smem_addr(smem + C::kOffK);
      const uint32_t sV = smem_addr(smem + C::kOffV);
      const uint32_t tS = tmem + 256 * x, tO = tS + 128;
      int cnt = 0;  // key tiles this query tile has finished
      bool ok = mbar_wait(&q_full, 0, &abort_flag, p.status, 201);
      int u = 0;
      for (int j = tiles.next(0); ok && j < tiles.end(); j = tiles.next(j + 1), ++u) {
        const int st = u % C::kStages;
        const uint32_t ph = (u / C::kStages) & 1;
        const bool vis = x == 0 ? tiles.vis_a(j) : tiles.vis_b(j);
        // Each issuer waits for the stage's load even when its tile does not
        // see key tile j: a commit made without it could run a whole ring ahead
        // and count toward the stage's current phase.
        ok = mbar_wait(&k_full[st], ph, &abort_flag, p.status, 202);
        if (!ok) break;
        if (vis) {
          // S_x = Q_x K_j^T, after x's previous P V (its P sits in the S columns)
          if (cnt > 0) ok = mbar_wait(&o_done[x], (cnt - 1) & 1, &abort_flag, p.status, 203 + x);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dK = sdesc_sw128(sK + st * C::kTileBytes, 16, 1024);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = ((ks >> 2) * C::kChunkBytes + (ks & 3) * 32) >> 4;
            mma_ss(tS, dQx + off, dK + off, idesc_qk, ks > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[x]);
        }
        mma_commit(&k_empty[st]);
        ok = mbar_wait(&v_full[st], ph, &abort_flag, p.status, 207);
        if (!ok) break;
        if (vis) {
          // O_x += P_x V_j, P_x read from TMEM (packed, 8 columns per 16 keys):
          // keys [0, 64) as soon as the softmax has written them, then the rest
          const uint64_t dV = sdesc_sw128(sV + st * C::kTileBytes, C::kChunkBytes, 1024);
          ok = mbar_wait(&p_half[x], cnt & 1, &abort_flag, p.status, 209 + x);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts(tO, tS + ks * 8, dV + ks * (2048 >> 4), idesc_pv, (cnt > 0 || ks > 0) ? 1u : 0u);
          ok = mbar_wait(&p_full[x], cnt & 1, &abort_flag, p.status, 205 + x);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 4; ks < 8; ++ks)
            mma_ts(tO, tS + ks * 8, dV + ks * (2048 >> 4), idesc_pv, 1u);
          mma_commit(&o_done[x]);
          ++cnt;
        }
        mma_commit(&v_empty[st]);
      }
      // all MMAs issued by this thread are complete once its drain flips
      mma_commit(&drain[x]);
      mbar_drain(&drain[x], 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;  // query tile: 0 = A, 1 = B
    const int qt = x == 0 ? qa : qb;
    const int row = qt * 128 + (tid & 127);
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 256 * x + lane_off, tO = tmem + 256 * x + 128 + lane_off;
    float m = -INFINITY, l = 0.f;
    int n = 0;
    bool ok = true;
    const bool live_tile = x == 0 || has_b;
    // additive bias: this row's [N] bias (nullptr past the end of the sequence)
    const bool bias_on = kExtra && p.bias != nullptr;
    const float* brow = (bias_on && row < p.N) ? p.bias + row_offset(p.lb, b, hd, row) : nullptr;
    if (live_tile) {
      int u = 0;  // key tiles either tile sees, in order
      for (int j = tiles.next(0); j < tiles.end(); j = tiles.next(j + 1), ++u) {
        // A's turn for key tile u comes after B's for u - 1, B's after A's for
        // u (each turn barrier's next phase needs this warpgroup's own next
        // pass, so no waiter can fall a phase behind).  Without a tile B, A
        // runs on its own.
        const bool vis = x == 0 ? tiles.vis_a(j) : tiles.vis_b(j);
        // dropout: this row's keep bits of the tile, drawn before the turn and S
        // are waited for (while the other warpgroup's softmax runs)
        uint32_t kbits[4] = {~0u, ~0u, ~0u, ~0u};
        if constexpr (kExtra) {
          if (vis && p.drop.t) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              kbits[c] = keep_bits_of_row(p.drop, (uint32_t)bh, row, j * 128 + 32 * c);
          }
        }
        if (C::kTurns && has_b && (x == 1 || u > 0)) {
          ok = mbar_wait_warp(&turn[x], (x == 1 ? u : u - 1) & 1, &abort_flag, p.status, 305 + x);
          if (!ok) break;
        }
        if (vis) {
          ok = mbar_wait_warp(&s_full[x], n & 1, &abort_flag, p.status, 301 + x);
          if (!ok) break;
          tc_fence_after();
          softmax_tile<kExtra>(tS, tO, D / 32, j * 128, kv_limit, row, p.causal != 0,
                               p.scale_log2, n == 0, m, l, &p_half[x], kbits, bias_on, brow,
                               p.N);
          tc_fence_before();
          mbar_arrive_warp(&p_full[x]);
          ++n;
        }
        if (C::kTurns && has_b) mbar_arrive_warp(&turn[x ^ 1]);  // the other tile's turn
      }
    }
    // ------------------------------------------------------------ epilogue
    if (ok && live_tile) {
      bool have = n > 0;
      if (have) {
        have = mbar_wait_warp(&o_done[x], (n - 1) & 1, &abort_flag, p.status, 304);
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
  if (warp == C::kIssuerWarp0) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int kTiles>
cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t s) {
  using C = FwdCfg<D, kTiles>;
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
  p.pairs = kTiles == 2 ? (p.T + 1) / 2 : p.T;
  // the work order holds query tiles at [0, T) and pairs of them at [2T, ...)
  p.order = p.block_mask && a.tile_order ? a.tile_order + (kTiles == 2 ? 2 * p.T : 0) : nullptr;
  p.BH = BH;
  p.group = grid_group_heads(a.B, a.H, a.N, a.d, a.causal);
  p.scale_log2 = a.scale * kLog2e;
  p.causal = a.causal;
  p.status = a.status;
  p.drop = a.drop;
  p.bias = a.bias;
  p.lb = a.lb;
  auto kernel = (a.drop.t || a.bias) ? fa_fwd_kernel<D, true, kTiles> : fa_fwd_kernel<D, false, kTiles>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.pairs * BH);
  return launch_pdl(kernel, grid, dim3(C::kThreads), C::kSmem, s, mq, mk, mv, p);
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t s) {
  if (a.d == 64 && !a.drop.t && !a.bias) return launch_fwd64_bf16(a, s);
  if (a.d == 128) return launch_fwd128s_bf16(a, s);
  return a.d == 64 ? launch_fwd_d<64, 1>(a, s) : launch_fwd_d<128, 2>(a, s);
}

}  // namespace fa
