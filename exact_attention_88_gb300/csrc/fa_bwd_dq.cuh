// Backward pass of exact attention, dQ, on sm_103a tensor cores: one CTA owns
// a 128-row query tile Q_i of one (batch, head), walks the key tiles K_j, V_j
// it can see, recomputes P from Q, K and the saved lse ("FlashAttention: Fast
// and Memory-Efficient Exact Attention with IO-Awareness", summary page, "Key
// ideas: recomputation in the backward pass") and accumulates
//   dQ_i = scale sum_j dS_ij K_j,  dS = P o (dP - D),  dP = dO V^T
// in TMEM.  Each dQ row is owned by one CTA, so it needs no atomics and the
// result does not depend on scheduling.  (The gradient formulas are the
// textbook derivative of the definition; the pages do not print them.)
//
// Query rows sit on the TMEM lanes, so lse and D are one scalar per thread.
// TMEM columns: S [0,128), dP_0 [128,256) and dP_1 [256,384) (dP_u alternates
// between them; once the math has read dP_u, packed bf16 dS_u goes over its
// first half), dQ accumulator [384, 384+d).  Per key tile u the math computes
// P_u from S_u (kept in registers), then dS_u; the tensor core work is
//   S_{u+1} = Q K_{u+1}^T   as soon as the math has read S_u
//   dP_{u+2} = dO V_{u+2}^T once dQ_u has read dS_u from that dP buffer
//   dQ += dS_u K_u          A = dS_u from TMEM, B = K_u (MN-major)
// so every MMA the math waits for was issued about a key tile earlier.
//
// Roles (640 threads): warps 0-15 are four math warpgroups -- warpgroup w owns
// key columns [32w, 32w+32) of S / dP and d columns [w d/4, (w+1) d/4) of the
// dQ read-out; warp 16 is the TMA producer; warps 17, 18, 19 issue S, dP and
// dQ (one thread each).
//
// Inputs are read through 4-D TMA descriptors with their own strides; dQ is
// stored through its strides.  A block-sparse CTA copies its row of the tile
// mask into a shared-memory bitmap first.  The kExtra variant adds dropout
// (a row's 32 keep bits of a key tile drawn before S is waited for; dS takes
// the dropped form of dP) and an additive bias (the row's 32 bias values read
// before S is waited for, added to the scaled scores).
//
// This header holds the CTA body; the kernels that run it are in the .cu files
// (the kernel of its own and the combined backward kernel).
#pragma once
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

template <int D>
struct DqCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kChunks = D / 64;
  static constexpr int kKStages = 3;        // K_j lives from S_j to dQ_j: one tile longer than V_j
  static constexpr int kVStages = 2;
  static constexpr int kPrefetchTiles = 4;  // L2 prefetch distance (key tiles)
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTileBytes;
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kSmem = kOffV + kVStages * kTileBytes + 1024;
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 384;  // dP_b at kColDP + 128 b
  static constexpr int kMathWarps = 16;
  static constexpr int kThreads = kMathWarps * 32 + 128;  // + producer, three MMA issuers
  static constexpr int kDSlice = D / 4;  // d columns per warpgroup in the read-out
  // V stage u % kVStages is also dP buffer u & 1 (two buffers of 128 columns
  // between kColDP and kColDQ)
  static_assert(kVStages == 2 && kColDP + 2 * 128 == kColDQ && kColDQ + D <= kTmemCols,
                "dP is double-buffered by the V stage");
};

struct DqParams {
  const float* lse;
  const float* Dvec;
  __nv_bfloat16* dq;
  Layout ldq;
  DropParams drop;
  const float* bias;  // additive score bias or nullptr
  Layout lb;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  const int32_t* order;  // block-sparse work order (query tiles) or nullptr
  int H, N, T, BH;
  int group;  // heads per group of the grid order
  float scale, scale_log2;
  int causal;
  int* status;
};

// Key tiles j that query tile qi sees: j < jend (causal diagonal, key
// padding, end of sequence), block-mask row qi (as a shared-memory bitmap;
// nullptr: no block mask).
struct KTileIter {
  const uint32_t* bits;
  int jend;
  __device__ int next(int j) const { return bits ? next_tile_bit(bits, j, jend) : j; }
};

template <int D, bool kExtra>
__device__ __forceinline__ void dq_cta(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                       const CUtensorMap& tmV, const CUtensorMap& tmDO, const DqParams& p, int cta) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t q_full, s_full, s_free, drain, drain_s, drain_p;
  // ds_ready[b]: dS of the key tile whose dP is in buffer b is written (over
  // that buffer).  dp_full[b]: dP of the key tile in V stage b (= dP buffer b)
  // is done; it frees the stage too.  dq_done[s]: dQ of the key tile in K
  // stage s is done; it frees the stage and the dP buffer that held its dS.
  // One commit each per key tile; per-buffer / per-stage barriers keep every
  // waiter within one phase (the next phase of each needs that waiter's own
  // progress first).
  __shared__ uint64_t ds_ready[2];
  __shared__ uint64_t k_full[C::kKStages], dq_done[C::kKStages];
  __shared__ uint64_t v_full[C::kVStages], dp_full[C::kVStages];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  uint32_t* const mask_bits = tile_mask_bitmap();  // block-mask row qi

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int order, bh;
  grid_order(cta, p.BH, p.T, p.group, &order, &bh);
  // causal: the last query tiles see the most keys: first; a block-sparse
  // work order lists the query tiles by their visible key tiles
  const int qi = ordered_tile(p.order, order, p.T, p.T - 1 - order);
  const int b = bh / p.H;
  const int hd = bh - b * p.H;
  int kv_limit = p.N;
  if (p.kv_len) kv_limit = max(0, min(p.kv_len[b], p.N));
  const int jkv = (kv_limit + 127) / 128;
  if (p.block_mask) build_tile_bitmap(mask_bits, p.block_mask + (size_t)qi * p.T, 1, p.T);
  const KTileIter ktiles{p.block_mask ? mask_bits : nullptr, p.causal ? min(jkv, qi + 1) : jkv};

  if (tid == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&s_full, 1);
    mbar_init(&s_free, C::kMathWarps);  // one arrival per math warp
    mbar_init(&drain, 1);
    mbar_init(&drain_s, 1);
    mbar_init(&drain_p, 1);
    for (int x = 0; x < 2; ++x) mbar_init(&ds_ready[x], C::kMathWarps);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&dq_done[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&dp_full[s], 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMathWarps + 1) tmem_alloc(&tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  pdl_launch_dependents();  // TMEM held: the next kernel may become resident
  const int jfirst = ktiles.next(0);  // after the barrier: the bitmap is complete
  const bool any = jfirst < ktiles.jend;

  if (warp == C::kMathWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && any) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmDO);
      mbar_expect_tx(&q_full, 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_4d(&tmQ, &q_full, smem + C::kOffQ + c * C::kChunkBytes, c * 64, qi * 128, hd, b);
        tma_load_4d(&tmDO, &q_full, smem + C::kOffDO + c * C::kChunkBytes, c * 64, qi * 128, hd, b);
      }
      int jpf = jfirst, npf = 0;
      auto prefetch_upto = [&](int count) {
        for (; npf < count && jpf < ktiles.jend; ++npf, jpf = ktiles.next(jpf + 1))
          for (int c = 0; c < C::kChunks; ++c) {
            tma_prefetch_4d(&tmK, c * 64, jpf * 128, hd, b);
            tma_prefetch_4d(&tmV, c * 64, jpf * 128, hd, b);
          }
      };
      prefetch_upto(C::kPrefetchTiles);
      int kcount[C::kKStages] = {}, vcount[C::kVStages] = {};
      int u = 0;
      for (int j = jfirst; j < ktiles.jend; j = ktiles.next(j + 1), ++u) {
        prefetch_upto(u + 1 + C::kPrefetchTiles);
        const int ks = u % C::kKStages, vs = u % C::kVStages;
        if (!mbar_wait(&dq_done[ks], ((u / C::kKStages) & 1) ^ 1, &abort_flag, p.status, 701))
          break;
        mbar_expect_tx(&k_full[ks], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(&tmK, &k_full[ks], smem + C::kOffK + ks * C::kTileBytes + c * C::kChunkBytes,
                      c * 64, j * 128, hd, b);
        ++kcount[ks];
        if (!mbar_wait(&dp_full[vs], ((u / C::kVStages) & 1) ^ 1, &abort_flag, p.status, 702))
          break;
        mbar_expect_tx(&v_full[vs], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(&tmV, &v_full[vs], smem + C::kOffV + vs * C::kTileBytes + c * C::kChunkBytes,
                      c * 64, j * 128, hd, b);
        ++vcount[vs];
      }
      // every issued copy must have landed before the CTA may exit
      mbar_drain(&q_full, 0);
      for (int s = 0; s < C::kKStages; ++s)
        if (kcount[s]) mbar_drain(&k_full[s], (kcount[s] - 1) & 1);
      for (int s = 0; s < C::kVStages; ++s)
        if (vcount[s]) mbar_drain(&v_full[s], (vcount[s] - 1) & 1);
    }
  } else if (warp >= C::kMathWarps + 1) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per MMA kind (an MMA costs its issuing thread about as
    // long as the tensor core takes to run it, so a thread waiting on one
    // dependency would starve the others):
    //   warp 17: S_u    -- after the math has read S_{u-1} (s_free)
    //   warp 18: dP_u   -- after dQ_{u-2} has read the dS in buffer u & 1
    //   warp 19: dQ_u   -- after the math has written dS_u (ds_ready)
    const int role = warp - (C::kMathWarps + 1);
    if (lane == 0 && any) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);  // S, dP
      constexpr uint32_t idesc_dq = idesc_bf16(128, D, false, true);    // dQ (A in TMEM)
      // operand descriptors built once; a K step adds its byte offset >> 4
      // to the start-address field (all buffers lie below 256 KB: no carry)
      const uint64_t dQ_k = sdesc_sw128(smem_addr(smem + C::kOffQ), 16, 1024);
      const uint64_t dDO_k = sdesc_sw128(smem_addr(smem + C::kOffDO), 16, 1024);
      const uint32_t sK = smem_addr(smem + C::kOffK), sV = smem_addr(smem + C::kOffV);
      bool ok = true;
      int u = 0;
      if (role == 0) {
        ok = mbar_wait(&q_full, 0, &abort_flag, p.status, 800);
        for (int j = jfirst; ok && j < ktiles.jend; j = ktiles.next(j + 1), ++u) {
          const int ks = u % C::kKStages;
          if (u > 0) ok = mbar_wait(&s_free, (u - 1) & 1, &abort_flag, p.status, 801);
          if (ok) ok = mbar_wait(&k_full[ks], (u / C::kKStages) & 1, &abort_flag, p.status, 802);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dK_k = sdesc_sw128(sK + ks * C::kTileBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
            mma_ss(tmem + C::kColS, dQ_k + off, dK_k + off, idesc_s, kk > 0);
          }
          mma_commit(&s_full);
        }
      } else if (role == 1) {
        ok = mbar_wait(&q_full, 0, &abort_flag, p.status, 803);
        for (int j = jfirst; ok && j < ktiles.jend; j = ktiles.next(j + 1), ++u) {
          const int vs = u % C::kVStages;  // = dP buffer
          if (u >= 2)
            ok = mbar_wait(&dq_done[(u - 2) % C::kKStages], ((u - 2) / C::kKStages) & 1,
                           &abort_flag, p.status, 804);
          if (ok) ok = mbar_wait(&v_full[vs], (u / C::kVStages) & 1, &abort_flag, p.status, 805);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dV_k = sdesc_sw128(sV + vs * C::kTileBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
            mma_ss(tmem + C::kColDP + 128 * vs, dDO_k + off, dV_k + off, idesc_s, kk > 0);
          }
          mma_commit(&dp_full[vs]);
        }
      } else {
        // dQ += dS_u K_u: dS_u packed in the first half of dP buffer u & 1
        // (warpgroup w's keys [32w, 32w+32) in columns [32w, 32w+16))
        for (int j = jfirst; ok && j < ktiles.jend; j = ktiles.next(j + 1), ++u) {
          const int ks = u % C::kKStages;
          ok = mbar_wait(&k_full[ks], (u / C::kKStages) & 1, &abort_flag, p.status, 806);
          if (ok) ok = mbar_wait(&ds_ready[u & 1], (u >> 1) & 1, &abort_flag, p.status, 807);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dK_mn = sdesc_sw128(sK + ks * C::kTileBytes, C::kChunkBytes, 1024);
          const uint32_t tA = tmem + C::kColDP + 128 * (u & 1);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::kColDQ, tA + 32 * (kk >> 1) + 8 * (kk & 1), dK_mn + kk * (2048 >> 4),
                   idesc_dq, (u > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&dq_done[ks]);
        }
      }
      // each issuer's MMAs are complete once its drain barrier flips; the last
      // dQ follows every S and dP (the math waited for both before its dS), so
      // `drain` alone tells the math that all are done
      uint64_t* my_drain = role == 0 ? &drain_s : role == 1 ? &drain_p : &drain;
      mma_commit(my_drain);
      mbar_drain(my_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ math warpgroups
    const int wg = warp >> 2;
    const int tq = tid & 127;  // TMEM lane: query row of the tile
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int q = qi * 128 + tq;
    const int col0 = wg * 32;  // this warpgroup's key columns
    float nl2 = -INFINITY, nd = 0.f;  // -lse2 (rows with no visible key: P = 0), -D
    if (q < p.N) {
      const float l = p.lse[(size_t)bh * p.N + q];
      if (l != -INFINITY) nl2 = -l * kLog2e;
      nd = -p.Dvec[(size_t)bh * p.N + q];
    }
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2), nl22 = make_float2(nl2, nl2);
    // additive bias: this query row's bias (nullptr past the end of the sequence)
    const bool bias_on = kExtra && p.bias != nullptr;
    const float* brow = (bias_on && q < p.N) ? p.bias + row_offset(p.lb, b, hd, q) : nullptr;
    const float2 sc2 = make_float2(p.scale, p.scale), nd2 = make_float2(nd, nd);
    int u = 0;
    bool ok = true;
    uint32_t keep_next = ~0u;  // dropout: the first key tile's keep bits
    if (kExtra && p.drop.t && jfirst < ktiles.jend)
      keep_next = keep_bits_of_row(p.drop, (uint32_t)bh, q, jfirst * 128 + col0);
    for (int j = jfirst; j < ktiles.jend; j = ktiles.next(j + 1), ++u) {
      const int x = u & 1;  // dP buffer
      const uint32_t tS = tmem + C::kColS + lane_off + col0;
      const uint32_t tP = tmem + C::kColDP + 128 * x + lane_off + col0;
      // keys [key0, key0 + 32) of this warpgroup; visible: key < kv_limit and,
      // causal, key <= q
      const int key0 = j * 128 + col0;
      // dropout: keep bits of the 32 keys (all set without dropout), drawn
      // during the previous key tile; bias: the 32 keys' bias, times log2(e), in
      // pf, read while S is computed
      const uint32_t keep = kExtra ? keep_next : 0u;
      float pf[32];
      if (kExtra && bias_on) load_bias_row<32>(brow, key0, p.N, pf);
      ok = mbar_wait_warp(&s_full, u & 1, &abort_flag, p.status, 901);
      if (!ok) break;
      tc_fence_after();
      int lim = kv_limit - key0;
      if (p.causal) lim = min(lim, q - key0 + 1);
      const bool partial = lim < 32;
      uint32_t rs_all[32];
      FA_TMEM_LD32_SYNC(tS, rs_all);
      // S_u is in registers: S_{u+1} may overwrite it while the exponentials run
      tc_fence_before();
      mbar_arrive_warp(&s_free);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t* rs = rs_all + 16 * h;
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          float2 t = fma2(make_float2(__uint_as_float(rs[e]), __uint_as_float(rs[e + 1])), c2, nl22);
          if (kExtra && bias_on) t = add2(t, make_float2(pf[16 * h + e], pf[16 * h + e + 1]));
          pf[16 * h + e] = ex2(t.x);
          pf[16 * h + e + 1] = ex2(t.y);
        }
      }
      if (partial) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (e >= lim) pf[e] = 0.f;
      }
      // dropout: the next key tile's keep bits, drawn while dP is computed
      if (kExtra && p.drop.t) {
        const int jn = ktiles.next(j + 1);
        keep_next = jn < ktiles.jend ? keep_bits_of_row(p.drop, (uint32_t)bh, q, jn * 128 + col0)
                                     : ~0u;
      }
      ok = mbar_wait_warp(&dp_full[x], (u >> 1) & 1, &abort_flag, p.status, 902);
      if (!ok) break;
      tc_fence_after();
      uint32_t dsp[16];
      uint32_t rp_all[32];
      FA_TMEM_LD32_SYNC(tP, rp_all);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t* rp = rp_all + 16 * h;
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float2 dpv = make_float2(__uint_as_float(rp[e]), __uint_as_float(rp[e + 1]));
          float2 t;
          if constexpr (kExtra) {
            // dS = P o (Z o dP / (1 - p) - D): dropped entries keep only -D
            const int c = 16 * h + e;
            const float2 zr = make_float2(((keep >> c) & 1u) ? p.drop.rp : 0.f,
                                          ((keep >> (c + 1)) & 1u) ? p.drop.rp : 0.f);
            t = fma2(dpv, zr, nd2);
          } else {
            t = add2(dpv, nd2);
          }
          const float2 dsv = mul2(mul2(make_float2(pf[16 * h + e], pf[16 * h + e + 1]), sc2), t);
          dsp[8 * h + e / 2] = pack_bf16(dsv.x, dsv.y);
        }
      }
      // packed dS of keys [col0, col0 + 32) over dP columns [col0, col0 + 16),
      // which this thread has read
      FA_TMEM_ST16(tP, dsp);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&ds_ready[x]);
    }
    // ------------------------------------------------------------ epilogue
    // `drain` completes once, after the issuer's last MMA: unlike the per-tile
    // barriers, whose earlier phases may still be pending here, it cannot alias
    bool have = false;
    if (__all_sync(0xffffffffu, ok && !abort_flag) && u > 0)
      have = mbar_wait_warp(&drain, 0, &abort_flag, p.status, 903);
    if (__all_sync(0xffffffffu, !abort_flag)) {  // warp-uniform: TMEM loads below
      tc_fence_after();
      uint32_t r[C::kDSlice];
      if (have) {
        if constexpr (C::kDSlice == 32) {
          FA_TMEM_LD32_SYNC(tmem + C::kColDQ + lane_off + wg * C::kDSlice, r);
        } else {
          FA_TMEM_LD16_SYNC(tmem + C::kColDQ + lane_off + wg * C::kDSlice, r);
        }
      } else {
#pragma unroll
        for (int e = 0; e < C::kDSlice; ++e) r[e] = 0u;  // no visible key: dQ = 0
      }
      if (q < p.N) {
        uint4* dst = reinterpret_cast<uint4*>(p.dq + row_offset(p.ldq, b, hd, q) + wg * C::kDSlice);
#pragma unroll
        for (int g = 0; g < C::kDSlice / 8; ++g) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(r[8 * g]), __uint_as_float(r[8 * g + 1]));
          w.y = pack_bf16(__uint_as_float(r[8 * g + 2]), __uint_as_float(r[8 * g + 3]));
          w.z = pack_bf16(__uint_as_float(r[8 * g + 4]), __uint_as_float(r[8 * g + 5]));
          w.w = pack_bf16(__uint_as_float(r[8 * g + 6]), __uint_as_float(r[8 * g + 7]));
          dst[g] = w;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kMathWarps + 1) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// The kernel parameters of a call (host).
inline DqParams make_dq_params(const BwdArgs& a) {
  DqParams p;
  p.lse = a.lse;
  p.Dvec = a.D;
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.ldq = a.ldq;
  p.drop = a.drop;
  p.bias = a.bias;
  p.lb = a.lb;
  p.kv_len = a.mask_kind == FA_MASK_KEY_PADDING ? a.kv_len : nullptr;
  p.block_mask = a.mask_kind == FA_MASK_BLOCK_SPARSE ? a.block_mask : nullptr;
  p.H = a.H;
  p.N = a.N;
  p.T = tiles_of(a.N, 128);
  p.BH = a.B * a.H;
  p.group = grid_group_heads(a.B, a.H, a.N, a.d, a.causal);
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.causal = a.causal;
  p.status = a.status;
  p.order = p.block_mask ? a.tile_order : nullptr;  // query tiles at [0, T)
  return p;
}

}  // namespace
}  // namespace fa
