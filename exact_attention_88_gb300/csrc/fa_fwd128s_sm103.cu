// Forward pass of exact attention at d = 128 on sm_103a tensor cores: one
// 128-row query tile per CTA, each key tile's softmax split between two
// warpgroups, and the scores double-buffered in TMEM ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", summary page, "Method":
// the softmax of a row is assembled from blocks, each with its own statistics
// m, l, and the partial results are merged by rescaling them to the common
// maximum; blog review, "Algorithm FlashAttention (Tiling)").
//
// Warpgroup h (h = 0, 1) owns keys [64h, 64h+64) of every key tile and keeps
// its own running statistics m_h, l_h and its own output accumulator O_h:
//   S(j)  = Q K_j^T               (N = 128: both halves)  into score buffer j & 1
//   P~_h  = 2^(c S_h(j) - m_h)    packed bf16 over the first 32 columns of half h
//   O_h   = O_h 2^(m_old - m_h) (lazily, when m_h grows by more than 8) + P~_h V_j,h
// and the epilogue merges the two halves as the d = 64 kernel does:
//   O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / l,  l = l_0 2^(m_0 - m) + l_1 2^(m_1 - m),
//   m = max(m_0, m_1),  lse = ln2 (m + log2 l).
// With two score buffers the tensor core computes S(j+1) while the softmax
// works on S(j); S(j+2) waits only for the P~ V of tile j, whose P~ sits in
// its buffer.  (With one buffer per query tile, as in the kernel that pairs two
// query tiles per CTA, the next S of a tile waits for the whole chain S ->
// softmax -> P~ V of the previous key tile.)  Each thread exponentiates 64
// scores per key tile, and both warpgroups' passes run at once.
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
// Roles (384 threads): warps 0-3 softmax of keys [0,64), warps 4-7 of keys
// [64,128) (thread = query row), warp 8 TMA producer (Q once; a K ring of 3
// and a V ring of 2, each K loaded one key tile ahead of its V), warp 9 issues
// S, warps 10 and 11 issue P~_0 V and P~_1 V (one thread each): the MMAs of a
// half's first 32 keys as soon as the softmax has written their P~ (p_half),
// the other two once the whole half is written (p_full).
// The barriers signalled per key tile (s_full, p_half, p_full, pv_done) are kept per
// score buffer: each has one phase per use of its buffer, and a buffer's next
// use needs its waiters' own progress first, so no waiter can fall two phases
// behind (a K load that arrives late cannot let a per-tile phase run ahead).
// With a block mask, a CTA walks only the key tiles its query tile sees (the
// mask row as a shared-memory bitmap), and a block-sparse work order may say
// which query tile each CTA takes.  This is the kernel of every d = 128
// call.  The kExtra variant
// adds dropout (a row's 64 keep bits of the half, drawn while the warpgroup waits
// for the tile's scores; dropped entries of P~ are zeroed in the packed P~ but
// counted in l, and O is scaled by 1 / (1 - p) at the end) and an additive bias
// (added to the scaled scores before the maximum).
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units: P~ stays below 2^8

struct Fwd128sCfg {
  static constexpr int D = 128;
  static constexpr int kChunkBytes = 128 * 128;   // 128 rows x 128 bytes (64 columns)
  static constexpr int kTileBytes = 128 * D * 2;  // one Q, K or V tile: two chunks
  static constexpr int kKStages = 3;              // K(j) is read by S(j), a tile ahead of V(j)
  static constexpr int kVStages = 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kSmem = kOffV + kVStages * kTileBytes + 1024;  // + alignment slack
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColO = 256;  // S_b at 128 b, O_h at kColO + 128 h
  static constexpr int kProducerWarp = 8;
  static constexpr int kSIssuerWarp = 9;
  static constexpr int kPvIssuerWarp0 = 10;
  static constexpr int kThreads = 32 * 12;
};

struct Fwd128sParams {
  __nv_bfloat16* o;
  Layout lo;
  float* lse;
  const int32_t* kv_len;
  int H, N, T, BH;
  int group;  // heads per group of the grid order
  float scale_log2;
  int causal;
  int* status;
  DropParams drop;
  const float* bias;  // additive score bias or nullptr
  Layout lb;
  const uint8_t* block_mask;  // T x T tile mask or nullptr
  const int32_t* order;       // block-sparse work order (query tiles) or nullptr
};

// Key tiles j < jend that a query tile sees: all of them, or those set in
// its block-mask row (a shared-memory bitmap).
struct KTiles {
  const uint32_t* bits;
  int jend;
  __device__ int next(int j) const { return bits ? next_tile_bit(bits, j, jend) : j; }
  __device__ int count() const {
    if (!bits) return jend;
    int c = 0;
    for (int w = 0; 32 * w < jend; ++w) {
      const int rest = jend - 32 * w;
      c += __popc(rest < 32 ? bits[w] & ((1u << rest) - 1u) : bits[w]);
    }
    return c;
  }
};

// Softmax of this warpgroup's 64 keys of one key tile for this thread's row:
// keys [0, lim) visible.  tS: the half's columns in the tile's score buffer,
// tO: the half's O columns (lane offset included).  O_h is rescaled only after
// the previous key tile's P~_h V has completed (pv_prev, pv_parity): the S of
// this tile may have been issued before it.  Returns false when that wait
// gave up.  kExtra: kbits holds the keep bits of the half's keys [0, 32) and
// [32, 64) (all set without dropout), brow this row's bias (nullptr past the
// end; bias_on warp-uniform), key0 the half's first key, n_keys the keys of a
// bias row.
// Keep bits of keys key0 + c, c = 0..63 (word c / 32, bit c % 32), of query row
// i: the bits keep_bits_of_row gives for key0 and key0 + 32, with all eight
// Philox calls in flight at once.
__device__ __forceinline__ void keep_bits64_of_row(const DropParams& d, uint32_t bh, int i, int key0,
                                                   uint32_t* out) {
  uint4 w[8];
#pragma unroll
  for (int g = 0; g < 8; ++g)
    w[g] = philox4x32_10((uint32_t)(key0 >> 3) + g, (uint32_t)i, bh, d.offset, d.k0, d.k1);
  out[0] = out[1] = 0u;
#pragma unroll
  for (int g = 0; g < 8; ++g) out[g >> 2] |= keep_bits8(w[g], d.t) << (8 * (g & 3));
}

template <bool kExtra>
__device__ __forceinline__ bool softmax_half128(uint32_t tS, uint32_t tO, int lim, float scale_log2,
                                                bool first, float& m, float& l, uint64_t* pv_prev,
                                                uint32_t pv_parity, volatile int* abort_flag,
                                                int* status, int site, uint64_t* p_half,
                                                const uint32_t* kbits, bool bias_on,
                                                const float* brow, int key0, int n_keys) {
  // the half-row's 64 scores, loaded once (one wait) for both passes
  uint32_t r[64];
  FA_TMEM_LD64_SYNC(tS, r);
  if (lim < 64) {
    mask32(r, lim);
    mask32(r + 32, lim - 32);
  }
  float exp_scale = scale_log2;  // multiplies what the exponent pass reads from r
  if (kExtra && bias_on) {
    // biased scores in log2 units: S scale log2(e) + bias log2(e)
    float bv[64];
    load_bias_row<64>(brow, key0, n_keys, bv);
#pragma unroll
    for (int e = 0; e < 64; ++e) r[e] = __float_as_uint(fmaf(__uint_as_float(r[e]), scale_log2, bv[e]));
    exp_scale = 1.f;
  }
  const float tmax = fmaxf(max32(r), max32(r + 32)) * exp_scale;
  const float m_new = fmaxf(m, tmax);
  const bool grow = m_new > m + kRescaleThreshold;  // true when m = -inf, m_new finite
  float alpha = 1.f;
  if (grow) {
    alpha = (m == -INFINITY) ? 0.f : ex2(m - m_new);
    m = m_new;
  }
  if (!first && __any_sync(0xffffffffu, grow)) {
    if (!mbar_wait_warp(pv_prev, pv_parity, abort_flag, status, site)) return false;
    tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      FA_TMEM_LD32_SYNC(tO + 32 * c, o);
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
      FA_TMEM_ST32(tO + 32 * c, o);
    }
  }
  const float nm = (m == -INFINITY) ? 0.f : -m;
  const float2 c2 = make_float2(exp_scale, exp_scale), nm2 = make_float2(nm, nm);
  float2 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float2(0.f, 0.f);
  // packed P~ of keys [32c, 32c + 32) over the half's columns [16c, 16c + 16),
  // already read; the first 32 keys are signalled as soon as they are written
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const int i = 32 * c + e;
      const float2 xx = fma2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), c2, nm2);
      float2 pv = make_float2(ex2(xx.x), ex2(xx.y));
      acc[(e >> 1) & 3] = add2(acc[(e >> 1) & 3], pv);  // l sums the undropped P~
      if constexpr (kExtra) {  // dropout (all bits set without it)
        if (!((kbits[c] >> e) & 1u)) pv.x = 0.f;
        if (!((kbits[c] >> (e + 1)) & 1u)) pv.y = 0.f;
      }
      pk[e >> 1] = pack_bf16(pv.x, pv.y);
    }
    FA_TMEM_ST16(tS + 16 * c, pk);
    if (c == 0) {
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(p_half);
    }
  }
  const float2 st = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
  l = l * alpha + (st.x + st.y);
  tmem_wait_st();
  return true;
}

template <bool kExtra>
__global__ void __launch_bounds__(Fwd128sCfg::kThreads, 1)
    fa_fwd128s_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const Fwd128sParams p) {
  using C = Fwd128sCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t q_full, drain[3];
  // per score buffer x: s_full (S in it), and per half h: p_half / p_full (P~_h
  // of the first 32 keys / of all 64 written, one arrival per warp of warpgroup
  // h), pv_done (P~_h V done: O_h is current and the half's columns of the
  // buffer are free)
  __shared__ uint64_t s_full[2], p_half[2][2], p_full[2][2], pv_done[2][2];
  __shared__ uint64_t k_full[C::kKStages], k_empty[C::kKStages];
  __shared__ uint64_t v_full[C::kVStages], v_empty[C::kVStages];
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
    for (int x = 0; x < 3; ++x) mbar_init(&drain[x], 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      for (int h = 0; h < 2; ++h) {
        mbar_init(&p_half[x][h], 4);
        mbar_init(&p_full[x][h], 4);
        mbar_init(&pv_done[x][h], 1);
      }
    }
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 2);  // one commit from each P~ V issuer
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kSIssuerWarp) tmem_alloc(&tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  pdl_launch_dependents();  // TMEM held: the next kernel may become resident
  // visible key tiles, counted after the barrier (the bitmap is complete); the
  // u-th of them is key tile tiles.next(...) walked from 0
  const int nt = tiles.count();

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      mbar_expect_tx(&q_full, C::kTileBytes);
      for (int c = 0; c < 2; ++c)
        tma_load_4d(&tmQ, &q_full, smem + C::kOffQ + c * C::kChunkBytes, c * 64, qi * 128, hd, b);
      int kcount[C::kKStages] = {}, vcount[C::kVStages] = {};
      auto load_k = [&](int u, int j) {
        const int st = u % C::kKStages;
        if (!mbar_wait(&k_empty[st], ((u / C::kKStages) & 1) ^ 1, &abort_flag, p.status, 2401))
          return false;
        mbar_expect_tx(&k_full[st], C::kTileBytes);
        for (int c = 0; c < 2; ++c)
          tma_load_4d(&tmK, &k_full[st], smem + C::kOffK + st * C::kTileBytes + c * C::kChunkBytes,
                      c * 64, j * 128, hd, b);
        ++kcount[st];
        return true;
      };
      auto load_v = [&](int u, int j) {
        const int st = u % C::kVStages;
        if (!mbar_wait(&v_empty[st], ((u / C::kVStages) & 1) ^ 1, &abort_flag, p.status, 2402))
          return false;
        mbar_expect_tx(&v_full[st], C::kTileBytes);
        for (int c = 0; c < 2; ++c)
          tma_load_4d(&tmV, &v_full[st], smem + C::kOffV + st * C::kTileBytes + c * C::kChunkBytes,
                      c * 64, j * 128, hd, b);
        ++vcount[st];
        return true;
      };
      int jk = tiles.next(0), jv = jk;  // key tiles of the next K and V loads
      bool ok = nt == 0 || load_k(0, jk);
      for (int u = 0; ok && u < nt; ++u) {
        if (u + 1 < nt) {
          jk = tiles.next(jk + 1);
          ok = load_k(u + 1, jk);
        }
        if (ok) ok = load_v(u, jv);
        jv = tiles.next(jv + 1);
      }
      // every issued copy must have landed before the CTA may exit
      mbar_drain(&q_full, 0);
      for (int s = 0; s < C::kKStages; ++s)
        if (kcount[s]) mbar_drain(&k_full[s], (kcount[s] - 1) & 1);
      for (int s = 0; s < C::kVStages; ++s)
        if (vcount[s]) mbar_drain(&v_full[s], (vcount[s] - 1) & 1);
    }
  } else if (warp == C::kSIssuerWarp) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
      const uint64_t dQ = sdesc_sw128(smem_addr(smem + C::kOffQ), 16, 1024);
      const uint32_t sK = smem_addr(smem + C::kOffK);
      bool ok = mbar_wait(&q_full, 0, &abort_flag, p.status, 2411);
      for (int u = 0; ok && u < nt; ++u) {
        const int st = u % C::kKStages, x = u & 1;
        ok = mbar_wait(&k_full[st], (u / C::kKStages) & 1, &abort_flag, p.status, 2412);
        // S(u) overwrites buffer x, where P~ of key tile u - 2 sits: both
        // halves' P~ V of that tile must be complete
        if (ok && u >= 2) ok = mbar_wait(&pv_done[x][0], ((u - 2) >> 1) & 1, &abort_flag, p.status, 2413);
        if (ok && u >= 2) ok = mbar_wait(&pv_done[x][1], ((u - 2) >> 1) & 1, &abort_flag, p.status, 2414);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dK = sdesc_sw128(sK + st * C::kTileBytes, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < C::D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * C::kChunkBytes + (ks & 3) * 32) >> 4;
          mma_ss(tmem + C::kColS + 128 * x, dQ + off, dK + off, idesc_qk, ks > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[x]);
        mma_commit(&k_empty[st]);
      }
      // all MMAs issued by this thread are complete once its drain flips
      mma_commit(&drain[0]);
      mbar_drain(&drain[0], 0);
    }
  } else if (warp >= C::kPvIssuerWarp0) {
    // ------------------------------------------------------------ P~_h V issuers
    const int h = warp - C::kPvIssuerWarp0;
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16(128, C::D, false, true);  // N = d, V MN-major
      const uint32_t sV = smem_addr(smem + C::kOffV);
      const uint32_t tO = tmem + C::kColO + 128 * h;
      bool ok = true;
      for (int u = 0; ok && u < nt; ++u) {
        const int st = u % C::kVStages, x = u & 1;
        ok = mbar_wait(&v_full[st], (u / C::kVStages) & 1, &abort_flag, p.status, 2415);
        if (ok) ok = mbar_wait(&p_half[x][h], (u >> 1) & 1, &abort_flag, p.status, 2418 + h);
        if (!ok) break;
        tc_fence_after();
        // O_h += P~_h V rows [64h, 64h + 64): P~ of 16 keys per 8 packed
        // columns; V row 64h + 16kk at byte 128 (64h + 16kk) of each chunk
        const uint64_t dV = sdesc_sw128(sV + st * C::kTileBytes, C::kChunkBytes, 1024);
        const uint32_t tP = tmem + C::kColS + 128 * x + 64 * h;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          mma_ts(tO, tP + 8 * kk, dV + (4 * h + kk) * (2048 >> 4), idesc_pv,
                 (u > 0 || kk > 0) ? 1u : 0u);
        ok = mbar_wait(&p_full[x][h], (u >> 1) & 1, &abort_flag, p.status, 2416 + h);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 2; kk < 4; ++kk)
          mma_ts(tO, tP + 8 * kk, dV + (4 * h + kk) * (2048 >> 4), idesc_pv, 1u);
        mma_commit(&pv_done[x][h]);
        mma_commit(&v_empty[st]);
      }
      mma_commit(&drain[1 + h]);
      mbar_drain(&drain[1 + h], 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int h = warp >> 2;  // key half
    const int tq = tid & 127;
    const int row = qi * 128 + tq;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + C::kColO + 128 * h + lane_off;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // additive bias: this row's [N] bias (nullptr past the end of the sequence)
    const bool bias_on = kExtra && p.bias != nullptr;
    const float* brow = (bias_on && row < p.N) ? p.bias + row_offset(p.lb, b, hd, row) : nullptr;
    int j = tiles.next(0);
    for (int n = 0; n < nt; ++n, j = tiles.next(j + 1)) {
      const int x = n & 1;
      // dropout: this row's keep bits of the half, drawn before the wait for S
      uint32_t kbits[2] = {~0u, ~0u};
      if constexpr (kExtra) {
        if (p.drop.t) keep_bits64_of_row(p.drop, (uint32_t)bh, row, j * 128 + 64 * h, kbits);
      }
      ok = mbar_wait_warp(&s_full[x], (n >> 1) & 1, &abort_flag, p.status, 2421 + h);
      if (!ok) break;
      tc_fence_after();
      // keys [key0, key0 + lim) of the half are visible from this row
      const int key0 = j * 128 + 64 * h;
      int lim = kv_limit - key0;
      if (p.causal) lim = min(lim, row - key0 + 1);
      // the previous key tile's P~_h V: buffer x ^ 1, that buffer's use (n - 1) / 2
      ok = softmax_half128<kExtra>(tmem + C::kColS + 128 * x + 64 * h + lane_off, tO, lim,
                                   p.scale_log2, n == 0, m, l, &pv_done[x ^ 1][h],
                                   ((n - 1) >> 1) & 1, &abort_flag, p.status, 2423 + h,
                                   &p_half[x][h], kbits, bias_on, brow, key0, p.N);
      if (!ok) break;
      tc_fence_before();
      mbar_arrive_warp(&p_full[x][h]);
    }
    // ------------------------------------------------------------ epilogue
    // both halves' accumulators must be complete before either is read; a
    // thread's commit covers its earlier MMAs, so the last tile's suffices
    bool have = ok && nt > 0;
    const int xl = (nt - 1) & 1;
    if (have) have = mbar_wait_warp(&pv_done[xl][0], ((nt - 1) >> 1) & 1, &abort_flag, p.status, 2425);
    if (have) have = mbar_wait_warp(&pv_done[xl][1], ((nt - 1) >> 1) & 1, &abort_flag, p.status, 2426);
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
      // dropout: the kept entries of P are scaled by 1 / (1 - p)
      const float inv = empty_row ? 0.f : (kExtra ? p.drop.rp : 1.f) / lt;
      const float w0 = a0 * inv, w1 = a1 * inv;
      // warpgroup h writes d columns [64h, 64h + 64) of the row
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const int col = 64 * h + 32 * c;
        uint32_t r0[32], r1[32];
        if (have) {
          FA_TMEM_LD32_SYNC(tmem + C::kColO + col + lane_off, r0);
          FA_TMEM_LD32_SYNC(tmem + C::kColO + 128 + col + lane_off, r1);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) r0[e] = r1[e] = 0u;
        }
        if (row < p.N) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + row_offset(p.lo, b, hd, row) + col);
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
        }
      }
      if (h == 0 && row < p.N)
        p.lse[(size_t)bh * p.N + row] = empty_row ? -INFINITY : (mm + __log2f(lt)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kSIssuerWarp) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace

cudaError_t launch_fwd128s_bf16(const FwdArgs& a, cudaStream_t s) {
  using C = Fwd128sCfg;
  const int BH = a.B * a.H;
  CUtensorMap mq, mk, mv;
  if (!encode_bhnd_map(&mq, a.q, a.lq, a.B, a.H, a.N, C::D, 128) ||
      !encode_bhnd_map(&mk, a.k, a.lk, a.B, a.H, a.N, C::D, 128) ||
      !encode_bhnd_map(&mv, a.v, a.lv, a.B, a.H, a.N, C::D, 128))
    return cudaErrorInvalidValue;
  Fwd128sParams p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lo = a.lo;
  p.lse = a.lse;
  p.kv_len = a.mask_kind == FA_MASK_KEY_PADDING ? a.kv_len : nullptr;
  p.H = a.H;
  p.N = a.N;
  p.T = tiles_of(a.N, 128);
  p.BH = BH;
  p.group = grid_group_heads(a.B, a.H, a.N, a.d, a.causal);
  p.scale_log2 = a.scale * kLog2e;
  p.causal = a.causal;
  p.status = a.status;
  p.drop = a.drop;
  p.bias = a.bias;
  p.lb = a.lb;
  p.block_mask = a.mask_kind == FA_MASK_BLOCK_SPARSE ? a.block_mask : nullptr;
  p.order = p.block_mask ? a.tile_order : nullptr;  // query tiles at [0, T)
  auto kernel = (a.drop.t || a.bias) ? fa_fwd128s_kernel<true> : fa_fwd128s_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(p.T * BH), dim3(C::kThreads), C::kSmem, s, mq, mk, mv, p);
}

}  // namespace fa
