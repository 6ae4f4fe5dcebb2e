// Backward pass of exact attention at d = 64, dQ, on sm_103a tensor cores: one
// CTA owns a 128-row query tile Q_i of one (batch, head), walks the key tiles
// K_j, V_j it can see, recomputes P from Q, K and the saved lse
// ("FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness", summary page, "Key ideas: recomputation in the backward
// pass") and accumulates
//   dQ_i = scale sum_j dS_ij K_j,  dS = P o (dP - D),  dP = dO V^T
// in TMEM.  Each dQ row is owned by one CTA, so it needs no atomics and the
// result does not depend on scheduling.  (The gradient formulas are the
// textbook derivative of the definition; the pages do not print them.)
// This is the kernel of d = 64 calls without dropout or a bias.
//
// Each key tile is taken in two steps of 64 keys, half h = 0, 1, so that a CTA
// needs 256 TMEM columns, 96 KB of shared memory and 384 threads and two CTAs
// share an SM: while one CTA's step waits on its chain, the other's runs.
// Query rows sit on the TMEM lanes; columns:
//   [0, 64)     S of the step (64 keys)
//   [64, 128), [128, 192)   dP of the step, alternating by step; once the math
//               has read it, packed bf16 dS goes over its first half
//   [192, 256)  dQ accumulator
// Per step s (key tile u, half h):
//   S_s = Q K_h^T            as soon as the math has read S_{s-1}
//   dP_s = dO V_h^T          once dQ_{s-2} has read the dS in that buffer
//   dQ += dS_s K_h           A = dS_s from TMEM, B = rows 64h.. of K_u
//
// Roles (384 threads): warps 0-7 are two math warpgroups -- warpgroup w owns
// key columns [32w, 32w+32) of each step and d columns [32w, 32w+32) of the
// dQ read-out; warp 8 is the TMA producer; warps 9, 10, 11 issue S, dQ and dP
// (one thread each).
//
// Inputs are read through 4-D TMA descriptors with their own strides; dQ is
// stored through its strides.  A block-sparse CTA copies its row of the tile
// mask into a shared-memory bitmap first.
//
// This header holds the CTA body; the kernels that run it are in the .cu files
// (the kernel of its own and the combined backward kernel).
#pragma once
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

struct Dq64Cfg {
  static constexpr int D = 64;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kKStages = 2;  // K_j lives from S to dQ
  static constexpr int kVStages = 2;
  static constexpr int kPrefetchTiles = 4;  // L2 prefetch distance (key tiles)
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTileBytes;
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kSmem = kOffV + kVStages * kTileBytes + 1024;
  static constexpr int kTmemCols = 256;
  static constexpr uint32_t kColS = 0, kColDP = 64, kColDQ = 192;  // dP_b at kColDP + 64 b
  static constexpr int kMathWarps = 8;
  static constexpr int kThreads = kMathWarps * 32 + 128;  // + producer, three MMA issuers
};

struct Dq64Params {
  const float* lse;
  const float* Dvec;
  __nv_bfloat16* dq;
  Layout ldq;
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
struct KTiles {
  const uint32_t* bits;
  int jend;
  __device__ int next(int j) const { return bits ? next_tile_bit(bits, j, jend) : j; }
};

__device__ __forceinline__ void dq64_cta(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                         const CUtensorMap& tmV, const CUtensorMap& tmDO, const Dq64Params& p, int cta) {
  using C = Dq64Cfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t q_full, s_full, s_free, drain, drain_s, drain_p;
  // Per step s (buffer b = s % 2): dp_full[b] (dP_s in buffer b), ds_ready[b]
  // (dS_s written over it by the 8 math warps), dq_done[b] (dQ_s has read it,
  // so dP_{s+2} may overwrite it).  Per stage: k_empty (dQ of the tile's
  // second half done: the last reader of K_u; S read it before), v_empty (dP
  // of the second half done).  Each completes once per step or tile, and each
  // next phase needs its waiter's own progress first.
  __shared__ uint64_t dp_full[2], ds_ready[2], dq_done[2];
  __shared__ uint64_t k_full[C::kKStages], k_empty[C::kKStages];
  __shared__ uint64_t v_full[C::kVStages], v_empty[C::kVStages];
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
  const KTiles ktiles{p.block_mask ? mask_bits : nullptr, p.causal ? min(jkv, qi + 1) : jkv};
  // 64-key steps of key tile j: the second is skipped when key padding hides
  // every key of it (no causal row of a tile the CTA sees loses a whole half).
  // Every role skips the same steps, and the step barriers count the steps
  // that run.
  auto steps_of = [&](int j) { return kv_limit > j * 128 + 64 ? 2 : 1; };

  if (tid == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&s_full, 1);
    mbar_init(&s_free, C::kMathWarps);  // one arrival per math warp
    mbar_init(&drain, 1);
    mbar_init(&drain_s, 1);
    mbar_init(&drain_p, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&dp_full[x], 1);
      mbar_init(&ds_ready[x], C::kMathWarps);
      mbar_init(&dq_done[x], 1);
    }
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
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
      tma_load_4d(&tmQ, &q_full, smem + C::kOffQ, 0, qi * 128, hd, b);
      tma_load_4d(&tmDO, &q_full, smem + C::kOffDO, 0, qi * 128, hd, b);
      int jpf = jfirst, npf = 0;
      auto prefetch_upto = [&](int count) {
        for (; npf < count && jpf < ktiles.jend; ++npf, jpf = ktiles.next(jpf + 1)) {
          tma_prefetch_4d(&tmK, 0, jpf * 128, hd, b);
          tma_prefetch_4d(&tmV, 0, jpf * 128, hd, b);
        }
      };
      prefetch_upto(C::kPrefetchTiles);
      int kcount[C::kKStages] = {}, vcount[C::kVStages] = {};
      int u = 0;
      for (int j = jfirst; j < ktiles.jend; j = ktiles.next(j + 1), ++u) {
        prefetch_upto(u + 1 + C::kPrefetchTiles);
        const int ks = u % C::kKStages, vs = u % C::kVStages;
        if (!mbar_wait(&k_empty[ks], ((u / C::kKStages) & 1) ^ 1, &abort_flag, p.status, 2001))
          break;
        mbar_expect_tx(&k_full[ks], C::kTileBytes);
        tma_load_4d(&tmK, &k_full[ks], smem + C::kOffK + ks * C::kTileBytes, 0, j * 128, hd, b);
        ++kcount[ks];
        if (!mbar_wait(&v_empty[vs], ((u / C::kVStages) & 1) ^ 1, &abort_flag, p.status, 2002))
          break;
        mbar_expect_tx(&v_full[vs], C::kTileBytes);
        tma_load_4d(&tmV, &v_full[vs], smem + C::kOffV + vs * C::kTileBytes, 0, j * 128, hd, b);
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
    //   warp 9:  S_s  -- after the math has read S_{s-1} (s_free)
    //   warp 10: dQ_s -- after the math has written dS_s (ds_ready)
    //   warp 11: dP_s -- after dQ_{s-2} has read the dS in buffer s % 2
    const int role = warp - (C::kMathWarps + 1);
    if (lane == 0 && any) {
      constexpr uint32_t idesc_64 = idesc_bf16(128, 64, false, false);  // S, dP of a step
      constexpr uint32_t idesc_dq = idesc_bf16(128, D, false, true);    // dQ (A in TMEM)
      // operand descriptors built once; a K step adds its byte offset >> 4 to
      // the start-address field (all buffers lie below 256 KB: no carry)
      const uint64_t dQ_k = sdesc_sw128(smem_addr(smem + C::kOffQ), 16, 1024);
      const uint64_t dDO_k = sdesc_sw128(smem_addr(smem + C::kOffDO), 16, 1024);
      const uint32_t sK = smem_addr(smem + C::kOffK), sV = smem_addr(smem + C::kOffV);
      bool ok = true;
      int u = 0, se = 0;  // key tiles, steps run
      if (role == 0) {
        ok = mbar_wait(&q_full, 0, &abort_flag, p.status, 2100);
        for (int j = jfirst; ok && j < ktiles.jend; j = ktiles.next(j + 1), ++u) {
          const int ks = u % C::kKStages;
          ok = mbar_wait(&k_full[ks], (u / C::kKStages) & 1, &abort_flag, p.status, 2101);
          const uint64_t dK_k = sdesc_sw128(sK + ks * C::kTileBytes, 16, 1024);
          const int nh = steps_of(j);
          for (int h = 0; h < nh && ok; ++h, ++se) {
            const int s = se;
            if (s > 0) ok = mbar_wait(&s_free, (s - 1) & 1, &abort_flag, p.status, 2102);
            if (!ok) break;
            tc_fence_after();
            // keys [64h, 64h + 64) of the tile: 64 x 128 bytes into it
            const uint64_t dKh = dK_k + ((uint32_t)(64 * 128 * h) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss(tmem + C::kColS, dQ_k + ((kk * 32) >> 4), dKh + ((kk * 32) >> 4), idesc_64,
                     kk > 0);
            mma_commit(&s_full);
          }
        }
      } else if (role == 2) {
        ok = mbar_wait(&q_full, 0, &abort_flag, p.status, 2103);
        for (int j = jfirst; ok && j < ktiles.jend; j = ktiles.next(j + 1), ++u) {
          const int vs = u % C::kVStages;
          ok = mbar_wait(&v_full[vs], (u / C::kVStages) & 1, &abort_flag, p.status, 2104);
          const uint64_t dV_k = sdesc_sw128(sV + vs * C::kTileBytes, 16, 1024);
          const int nh = steps_of(j);
          for (int h = 0; h < nh && ok; ++h, ++se) {
            const int s = se, x = s & 1;
            if (s >= 2) ok = mbar_wait(&dq_done[x], ((s - 2) >> 1) & 1, &abort_flag, p.status, 2105);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dVh = dV_k + ((uint32_t)(64 * 128 * h) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss(tmem + C::kColDP + 64 * x, dDO_k + ((kk * 32) >> 4), dVh + ((kk * 32) >> 4),
                     idesc_64, kk > 0);
            mma_commit(&dp_full[x]);
          }
          if (ok) mma_commit(&v_empty[vs]);  // both halves of V_u read
        }
      } else {
        // dQ += dS_s K_h: dS_s packed in the first half of dP buffer s % 2
        // (warpgroup w's keys [32w, 32w+32) in columns [32w, 32w+16)); B = rows
        // 64h + 16kk of K_u, d contiguous (MN-major)
        for (int j = jfirst; ok && j < ktiles.jend; j = ktiles.next(j + 1), ++u) {
          const int ks = u % C::kKStages;
          ok = mbar_wait(&k_full[ks], (u / C::kKStages) & 1, &abort_flag, p.status, 2106);
          const uint64_t dK_mn = sdesc_sw128(sK + ks * C::kTileBytes, C::kChunkBytes, 1024);
          const int nh = steps_of(j);
          for (int h = 0; h < nh && ok; ++h, ++se) {
            const int s = se, x = s & 1;
            ok = mbar_wait(&ds_ready[x], (s >> 1) & 1, &abort_flag, p.status, 2107);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tA = tmem + C::kColDP + 64 * x;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tmem + C::kColDQ, tA + 32 * (kk >> 1) + 8 * (kk & 1),
                     dK_mn + (4 * h + kk) * (2048 >> 4), idesc_dq, (s > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&dq_done[x]);
          }
          if (ok) mma_commit(&k_empty[ks]);  // dQ, the last reader of K_u, is done
        }
      }
      // each issuer's MMAs are complete once its drain barrier flips; the last
      // dQ follows every S and dP (the math waited for both before its dS), so
      // `drain` alone tells the math that all are done
      uint64_t* my_drain = role == 0 ? &drain_s : role == 2 ? &drain_p : &drain;
      mma_commit(my_drain);
      mbar_drain(my_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ math warpgroups
    const int wg = warp >> 2;
    const int tq = tid & 127;  // TMEM lane: query row of the tile
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int q = qi * 128 + tq;
    const int col0 = wg * 32;  // this warpgroup's key columns of a step
    float nl2 = -INFINITY, nd = 0.f;  // -lse2 (rows with no visible key: P = 0), -D
    if (q < p.N) {
      const float l = p.lse[(size_t)bh * p.N + q];
      if (l != -INFINITY) nl2 = -l * kLog2e;
      nd = -p.Dvec[(size_t)bh * p.N + q];
    }
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2), nl22 = make_float2(nl2, nl2);
    const float2 sc2 = make_float2(p.scale, p.scale), nd2 = make_float2(nd, nd);
    int u = 0, se = 0;  // key tiles, steps run
    bool ok = true;
    for (int j = jfirst; ok && j < ktiles.jend; j = ktiles.next(j + 1), ++u) {
      const int nh = steps_of(j);
#pragma unroll 1
      for (int h = 0; h < nh; ++h, ++se) {
        const int s = se, x = s & 1;
        const uint32_t tP = tmem + C::kColDP + 64 * x + lane_off + col0;
        // keys [key0, key0 + 32) of this warpgroup; visible: key < kv_limit and,
        // causal, key <= q
        const int key0 = j * 128 + 64 * h + col0;
        ok = mbar_wait_warp(&s_full, s & 1, &abort_flag, p.status, 2201);
        if (!ok) break;
        tc_fence_after();
        int lim = kv_limit - key0;
        if (p.causal) lim = min(lim, q - key0 + 1);
        uint32_t rs[32];
        FA_TMEM_LD32_SYNC(tmem + C::kColS + lane_off + col0, rs);
        // S_s is in registers: S_{s+1} may overwrite it while the exponentials run
        tc_fence_before();
        mbar_arrive_warp(&s_free);
        float pf[32];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 t = fma2(make_float2(__uint_as_float(rs[e]), __uint_as_float(rs[e + 1])), c2,
                                nl22);
          pf[e] = ex2(t.x);
          pf[e + 1] = ex2(t.y);
        }
        if (lim < 32) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e >= lim) pf[e] = 0.f;
        }
        ok = mbar_wait_warp(&dp_full[x], (s >> 1) & 1, &abort_flag, p.status, 2202);
        if (!ok) break;
        tc_fence_after();
        uint32_t rp[32];
        FA_TMEM_LD32_SYNC(tP, rp);
        uint32_t dsp[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 t = add2(make_float2(__uint_as_float(rp[e]), __uint_as_float(rp[e + 1])), nd2);
          const float2 dsv = mul2(mul2(make_float2(pf[e], pf[e + 1]), sc2), t);
          dsp[e / 2] = pack_bf16(dsv.x, dsv.y);
        }
        // packed dS of keys [col0, col0 + 32) over dP columns [col0, col0 + 16),
        // which this thread has read
        FA_TMEM_ST16(tP, dsp);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(&ds_ready[x]);
      }
    }
    // ------------------------------------------------------------ epilogue
    // `drain` completes once, after the issuer's last MMA
    bool have = false;
    if (__all_sync(0xffffffffu, ok && !abort_flag) && u > 0)
      have = mbar_wait_warp(&drain, 0, &abort_flag, p.status, 2203);
    if (__all_sync(0xffffffffu, !abort_flag)) {  // warp-uniform: TMEM loads below
      tc_fence_after();
      uint32_t r[32];
      if (have) {
        FA_TMEM_LD32_SYNC(tmem + C::kColDQ + lane_off + wg * 32, r);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = 0u;  // no visible key: dQ = 0
      }
      if (q < p.N) {
        uint4* dst = reinterpret_cast<uint4*>(p.dq + row_offset(p.ldq, b, hd, q) + wg * 32);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
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
inline Dq64Params make_dq64_params(const BwdArgs& a) {
  Dq64Params p;
  p.lse = a.lse;
  p.Dvec = a.D;
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.ldq = a.ldq;
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
