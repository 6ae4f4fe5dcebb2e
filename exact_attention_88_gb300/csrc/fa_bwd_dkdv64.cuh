// Backward pass of exact attention on sm_103a tensor cores at d = 64, dK and
// dV, with P recomputed on chip from Q, K and lse ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", summary page, "Key
// ideas: recomputation in the backward pass").  The gradient formulas are the
// textbook derivative of the definition (the pages do not print them): with
// S = scale Q K^T, P = exp(S - lse), D_i = rowsum(dO o O)_i,
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  dK = scale dS^T Q.
// This is the kernel of d = 64 calls without dropout or a bias.
//
// One CTA owns a 128-key tile K_j, V_j of one (batch, head) and walks the
// query tiles Q_i that can see it (causal: i >= j; block-sparse: mask[i][j])
// in steps of 64 query rows, half h = 0, 1 of each tile; two CTAs share an SM
// (256 TMEM columns, ≈100 KB of shared memory and 384 threads each), so that
// while one CTA's step waits on its chain S^T -> P^T -> dV -> next S^T the
// other's runs.  Keys sit on the TMEM lanes; columns:
//   [0, 64) dV     [64, 128) dK
//   [128, 192)     S^T_h = K_j Q_h^T of the step, then P^T (bf16, packed two
//                  per column: warpgroup w's 32 query columns in [32w, 32w+16))
//   [192, 256)     dP^T_h = V_j dO_h^T, then dS^T (packed the same way)
// Per step: S^T (issuer A, after the previous step's dV), dP^T (issuer C,
// after the previous step's dK), P^T and dS^T (math), dV += P^T dO_h and
// dK += dS^T Q_h (issuer B, A from TMEM).
//
// Roles (384 threads): warps 0-7 are two math warpgroups -- warpgroup w owns
// query columns [32w, 32w+32) of each step and d columns [32w, 32w+32) of the
// dK, dV read-out; warp 8 loads (TMA for K, V, Q, dO; plain loads for the
// statistics -lse2, -D of each query tile, kept in shared memory beside its Q
// stage); warps 9, 10 and 11 issue the MMAs (S^T; dV and dK; dP^T).
//
// Inputs are read through 4-D TMA descriptors with their own strides; dK, dV
// are stored through theirs.  A block-sparse CTA copies its column of the tile
// mask into a shared-memory bitmap first.
//
// This header holds the CTA body; the kernels that run it are in the .cu files
// (the kernel of its own and the combined backward kernel).
#pragma once
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

struct Bwd64Cfg {
  static constexpr int D = 64;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kChunks = D / 64;
  static constexpr int kQStages = 2;   // Q ring (Q_i lives from S^T to dK)
  static constexpr int kDOStages = 2;  // dO ring
  static constexpr int kPrefetchTiles = 4;  // L2 prefetch distance (query tiles)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;
  static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;
  static constexpr int kSmem = kOffDO + kDOStages * kTileBytes + 1024;
  static constexpr int kTmemCols = 256;
  static constexpr uint32_t kColDV = 0, kColDK = 64, kColS = 128, kColDP = 192;
  static constexpr int kMathWarps = 8;
  static constexpr int kThreads = kMathWarps * 32 + 128;  // + loader, three MMA issuers
  static constexpr int kDSlice = 32;  // d columns per warpgroup in the dK / dV read-out
};

struct Bwd64Params {
  const float* lse;
  const float* Dvec;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  Layout ldk, ldv;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  const int32_t* order;  // block-sparse work order (key tiles) or nullptr
  int H, N, T, BH;
  int group;  // heads per group of the grid order
  float scale, scale_log2;
  int causal;
  int* status;
};

// Query tiles i that see key tile kt: i in [ibegin, T), block-mask column kt
// (as a shared-memory bitmap; nullptr: no block mask).
struct QTiles {
  const uint32_t* bits;
  int T, ibegin;
  __device__ int first() const { return next(ibegin); }
  __device__ int next(int i) const { return bits ? next_tile_bit(bits, i, T) : i; }
};

// n fp32 values (TMEM words) stored as bf16.
__device__ __forceinline__ void store_row(__nv_bfloat16* dst, const uint32_t* r, int n) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  auto f = [&](int e) { return __uint_as_float(r[e]); };
  for (int g = 0; g < n / 8; ++g) {
    uint4 w;
    w.x = pack_bf16(f(8 * g), f(8 * g + 1));
    w.y = pack_bf16(f(8 * g + 2), f(8 * g + 3));
    w.z = pack_bf16(f(8 * g + 4), f(8 * g + 5));
    w.w = pack_bf16(f(8 * g + 6), f(8 * g + 7));
    d4[g] = w;
  }
}

__device__ __forceinline__ void dkdv64_cta(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                           const CUtensorMap& tmV, const CUtensorMap& tmDO, const Bwd64Params& p, int cta) {
  using C = Bwd64Cfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t kv_full, drain, drain_a, drain_c;
  // q_full[s]: Q_i and its statistics are in stage s (two arrivals: the TMA
  // transaction and the loader's statistics stores).  q_empty[s]: dK of the
  // tile's second half is done -- the last reader of Q_i and, through the
  // math's dS^T before it, of the statistics.  do_full / do_empty: dO_i, whose
  // two readers are dP^T (issuer C) and dV (issuer B).
  __shared__ uint64_t q_full[C::kQStages], q_empty[C::kQStages];
  __shared__ uint64_t do_full[C::kDOStages], do_empty[C::kDOStages];
  // per step (64 query rows): s_full (S^T in TMEM), s_free (its dV done),
  // dp_full, dp_free (its dK done), p_ready / ds_ready (P^T / dS^T written by
  // all 8 math warps).  Each completes once per step; a waiter can never fall
  // a phase behind, because each next phase needs that waiter's own progress.
  __shared__ uint64_t s_full, s_free, dp_full, dp_free, p_ready, ds_ready;
  __shared__ __align__(16) float s_nl2[C::kQStages][128];  // -lse2 of the stage's query rows
  __shared__ __align__(16) float s_nD[C::kQStages][128];   // -D
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  uint32_t* const mask_bits = tile_mask_bitmap();  // block-mask column kt

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int kt, bh;  // key tile (causal: low tiles have the most work: first)
  grid_order(cta, p.BH, p.T, p.group, &kt, &bh);
  kt = ordered_tile(p.order, kt, p.T, kt);  // block-sparse work order: by query tiles seen
  const int b = bh / p.H;
  const int hd = bh - b * p.H;
  int kv_limit = p.N;
  if (p.kv_len) kv_limit = max(0, min(p.kv_len[b], p.N));
  const bool keys_live = kt * 128 < kv_limit;  // else every key of the tile is padding
  if (!keys_live) {
    // every key of the tile is padding: its dK, dV rows are zero and no MMA
    // runs, so the CTA writes them and leaves before any set-up (key padding
    // leaves about a third of the key tiles dead at BERT's lengths)
    constexpr int kRowChunks = D / 8;  // 16-byte chunks of a row
    for (int e = tid; e < 2 * 128 * kRowChunks; e += blockDim.x) {
      const int which = e / (128 * kRowChunks), r = (e / kRowChunks) % 128, c = e % kRowChunks;
      const int key = kt * 128 + r;
      if (key < p.N) {
        __nv_bfloat16* row = which == 0 ? p.dv + row_offset(p.ldv, b, hd, key)
                                        : p.dk + row_offset(p.ldk, b, hd, key);
        reinterpret_cast<uint4*>(row)[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }
  if (p.block_mask) build_tile_bitmap(mask_bits, p.block_mask + kt, (size_t)p.T, p.T);
  const QTiles qtiles{p.block_mask ? mask_bits : nullptr, p.T, p.causal ? kt : 0};
  const int iend = keys_live ? p.T : 0;

  if (tid == 0) {
    mbar_init(&kv_full, 1);
    mbar_init(&drain, 1);
    mbar_init(&drain_a, 1);
    mbar_init(&drain_c, 1);
    mbar_init(&s_full, 1);
    mbar_init(&s_free, 1);
    mbar_init(&dp_full, 1);
    mbar_init(&dp_free, 1);
    mbar_init(&p_ready, C::kMathWarps);
    mbar_init(&ds_ready, C::kMathWarps);
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(&q_full[s], 2);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < C::kDOStages; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 2);
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

  if (warp == C::kMathWarps) {
    // ------------------------------------------------------------ loader
    if (iend > 0) {
      const size_t head_row0 = (size_t)bh * p.N;
      if (lane == 0) {
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        prefetch_tensormap(&tmDO);
        mbar_expect_tx(&kv_full, 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_4d(&tmK, &kv_full, smem + C::kOffK + c * C::kChunkBytes, c * 64, kt * 128, hd,
                      b);
          tma_load_4d(&tmV, &kv_full, smem + C::kOffV + c * C::kChunkBytes, c * 64, kt * 128, hd,
                      b);
        }
      }
      int qcount[C::kQStages] = {}, dcount[C::kDOStages] = {};
      // L2 prefetch of the Q / dO tiles a few query tiles ahead of their loads
      int ipf = qtiles.first(), npf = 0;
      auto prefetch_upto = [&](int count) {
        for (; npf < count && ipf < iend; ++npf, ipf = qtiles.next(ipf + 1))
          if (lane == 0)
            for (int c = 0; c < C::kChunks; ++c) {
              tma_prefetch_4d(&tmQ, c * 64, ipf * 128, hd, b);
              tma_prefetch_4d(&tmDO, c * 64, ipf * 128, hd, b);
            }
      };
      prefetch_upto(C::kPrefetchTiles);
      int it = 0;
      for (int i = qtiles.first(); i < iend; i = qtiles.next(i + 1), ++it) {
        const int qs = it % C::kQStages, ds = it % C::kDOStages;
        prefetch_upto(it + 1 + C::kPrefetchTiles);
        if (!mbar_wait_warp(&q_empty[qs], ((it / C::kQStages) & 1) ^ 1, &abort_flag, p.status,
                            1901))
          break;
        if (lane == 0) {
          mbar_expect_tx(&q_full[qs], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(&tmQ, &q_full[qs],
                        smem + C::kOffQ + qs * C::kTileBytes + c * C::kChunkBytes, c * 64, i * 128,
                        hd, b);
        }
        ++qcount[qs];
        // statistics of the tile's rows, in the form the math uses: -lse2
        // (rows with no visible key, lse = -inf, and rows past the end keep
        // -inf: P = 0) and -D
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = lane + 32 * k, q = i * 128 + r;
          float nl2 = -INFINITY, nd = 0.f;
          if (q < p.N) {
            const float l = p.lse[head_row0 + q];
            nl2 = l == -INFINITY ? -INFINITY : -l * kLog2e;
            nd = -p.Dvec[head_row0 + q];
          }
          s_nl2[qs][r] = nl2;
          s_nD[qs][r] = nd;
        }
        mbar_arrive_warp(&q_full[qs]);
        if (!mbar_wait_warp(&do_empty[ds], ((it / C::kDOStages) & 1) ^ 1, &abort_flag, p.status,
                            1902))
          break;
        if (lane == 0) {
          mbar_expect_tx(&do_full[ds], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(&tmDO, &do_full[ds],
                        smem + C::kOffDO + ds * C::kTileBytes + c * C::kChunkBytes, c * 64,
                        i * 128, hd, b);
        }
        ++dcount[ds];
      }
      // every issued copy must have landed before the CTA may exit
      if (lane == 0) {
        mbar_drain(&kv_full, 0);
        for (int s = 0; s < C::kQStages; ++s)
          if (qcount[s]) mbar_drain(&q_full[s], (qcount[s] - 1) & 1);
        for (int s = 0; s < C::kDOStages; ++s)
          if (dcount[s]) mbar_drain(&do_full[s], (dcount[s] - 1) & 1);
      }
    }
  } else if (warp > C::kMathWarps) {
    // ------------------------------------------------------------ MMA issuers
    //   A (warp 9):  S^T of each step -- gated by Q_i and by the previous
    //                step's dV (the reader of the P^T in the S^T columns)
    //   B (warp 10): dV and dK -- gated by the math (P^T, dS^T)
    //   C (warp 11): dP^T of each step -- gated by dO_i and by the previous
    //                step's dK (the reader of the dS^T in the dP^T columns)
    const int role = warp - C::kMathWarps - 1;  // 0: A, 1: B, 2: C
    if (lane == 0 && iend > 0) {
      constexpr uint32_t idesc_64 = idesc_bf16(128, 64, false, false);   // S^T, dP^T of a step
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, false, true);    // dV, dK
      const uint32_t sK = smem_addr(smem + C::kOffK), sV = smem_addr(smem + C::kOffV);
      const uint32_t sQ0 = smem_addr(smem + C::kOffQ), sDO0 = smem_addr(smem + C::kOffDO);
      // operand descriptors built once per buffer; a K step adds its byte
      // offset >> 4 to the start-address field (every buffer lies below 256 KB)
      const uint64_t dK_k = sdesc_sw128(sK, 16, 1024), dV_k = sdesc_sw128(sV, 16, 1024);
      bool ok = role == 1 || mbar_wait(&kv_full, 0, &abort_flag, p.status, 1701);  // K, V
      int it = 0;
      for (int i = qtiles.first(); ok && i < iend; i = qtiles.next(i + 1), ++it) {
        const int qs = it % C::kQStages, ds = it % C::kDOStages;
        const uint32_t sQ = sQ0 + qs * C::kTileBytes, sDO = sDO0 + ds * C::kTileBytes;
        if (role == 0) {
          ok = mbar_wait(&q_full[qs], (it / C::kQStages) & 1, &abort_flag, p.status, 1702);
          const uint64_t dQ_k = sdesc_sw128(sQ, 16, 1024);
          for (int h = 0; h < 2 && ok; ++h) {
            const int st = 2 * it + h;  // step
            if (st > 0) ok = mbar_wait(&s_free, (st - 1) & 1, &abort_flag, p.status, 1703);
            if (!ok) break;
            tc_fence_after();
            // S^T = K Q^T of query rows [64h, 64h + 64): 64 x 128 bytes into the tile
            const uint64_t dQh = dQ_k + ((uint32_t)(64 * 128 * h) >> 4);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              mma_ss(tmem + C::kColS, dK_k + ((ks * 32) >> 4), dQh + ((ks * 32) >> 4), idesc_64,
                     ks > 0);
            mma_commit(&s_full);
          }
        } else if (role == 2) {
          ok = mbar_wait(&do_full[ds], (it / C::kDOStages) & 1, &abort_flag, p.status, 1704);
          const uint64_t dDO_k = sdesc_sw128(sDO, 16, 1024);
          for (int h = 0; h < 2 && ok; ++h) {
            const int st = 2 * it + h;
            if (st > 0) ok = mbar_wait(&dp_free, (st - 1) & 1, &abort_flag, p.status, 1705);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dDOh = dDO_k + ((uint32_t)(64 * 128 * h) >> 4);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              mma_ss(tmem + C::kColDP, dV_k + ((ks * 32) >> 4), dDOh + ((ks * 32) >> 4), idesc_64,
                     ks > 0);
            mma_commit(&dp_full);
          }
          if (ok) mma_commit(&do_empty[ds]);  // this reader of dO_i is done
        } else {
          // dV += P^T dO_h and dK += dS^T Q_h: A from TMEM (warpgroup w's 32
          // query columns packed in columns [32w, 32w+16): K steps 2w, 2w+1),
          // B MN-major (K step ks of half h = rows 64h + 16ks: 2048 bytes per
          // 16 rows)
          ok = mbar_wait(&q_full[qs], (it / C::kQStages) & 1, &abort_flag, p.status, 1706);
          if (ok) ok = mbar_wait(&do_full[ds], (it / C::kDOStages) & 1, &abort_flag, p.status, 1707);
          const uint64_t dQ_mn = sdesc_sw128(sQ, C::kChunkBytes, 1024);
          const uint64_t dDO_mn = sdesc_sw128(sDO, C::kChunkBytes, 1024);
          for (int h = 0; h < 2 && ok; ++h) {
            const int st = 2 * it + h;
            ok = mbar_wait(&p_ready, st & 1, &abort_flag, p.status, 1708);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_ts(tmem + C::kColDV, tmem + C::kColS + 32 * (ks >> 1) + 8 * (ks & 1),
                     dDO_mn + (4 * h + ks) * (2048 >> 4), idesc_acc, (st > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&s_free);
            if (h == 1) mma_commit(&do_empty[ds]);  // this reader of dO_i is done
            ok = mbar_wait(&ds_ready, st & 1, &abort_flag, p.status, 1709);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_ts(tmem + C::kColDK, tmem + C::kColDP + 32 * (ks >> 1) + 8 * (ks & 1),
                     dQ_mn + (4 * h + ks) * (2048 >> 4), idesc_acc, (st > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&dp_free);
          }
          if (ok) mma_commit(&q_empty[qs]);
        }
      }
      // B's last dK follows every MMA of A and C (its last dV waited for the last
      // S^T through p_ready, its last dK for the last dP^T through ds_ready), so
      // `drain` alone tells the math that all are done
      uint64_t* my_drain = role == 0 ? &drain_a : role == 2 ? &drain_c : &drain;
      mma_commit(my_drain);
      mbar_drain(my_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ math warpgroups
    const int wg = warp >> 2;  // 0, 1
    const int tq = tid & 127;  // TMEM lane: key row of the tile
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int key = kt * 128 + tq;
    const bool key_live = key < kv_limit;
    const int col0 = wg * 32;  // this warpgroup's query columns of a step
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    const float2 sc2 = make_float2(p.scale, p.scale);
    int it = 0;
    bool ok = true;
    for (int i = qtiles.first(); i < iend; i = qtiles.next(i + 1), ++it) {
      const int qs = it % C::kQStages;
      // the statistics of the tile are in place with Q_i
      ok = mbar_wait_warp(&q_full[qs], (it / C::kQStages) & 1, &abort_flag, p.status, 1800);
      if (!ok) break;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const int st = 2 * it + h;
        const int q0 = i * 128 + 64 * h + col0;  // query row of column 0 of this thread's 32
        // ---- P^T = 2^(c S^T - lse2) for the warpgroup's 32 query columns
        ok = mbar_wait_warp(&s_full, st & 1, &abort_flag, p.status, 1801);
        if (!ok) break;
        tc_fence_after();
        uint32_t rs[32];
        FA_TMEM_LD32_SYNC(tmem + C::kColS + lane_off + col0, rs);
        float pf[32];
        const float* nl2 = &s_nl2[qs][64 * h + col0];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float4 L = *reinterpret_cast<const float4*>(nl2 + 4 * g);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 4 * g + 2 * u;
            const float2 x = fma2(make_float2(__uint_as_float(rs[e]), __uint_as_float(rs[e + 1])),
                                  c2, u ? make_float2(L.z, L.w) : make_float2(L.x, L.y));
            pf[e] = ex2(x.x);
            pf[e + 1] = ex2(x.y);
          }
        }
        // causal diagonal tiles and padded keys
        if (!key_live || (p.causal && key > q0)) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (!key_live || key > q0 + e) pf[e] = 0.f;
        }
        uint32_t pp[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) pp[e / 2] = pack_bf16(pf[e], pf[e + 1]);
        FA_TMEM_ST16(tmem + C::kColS + lane_off + col0, pp);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(&p_ready);
        // ---- dS^T = scale P^T o (dP^T - D), packed over dP^T
        ok = mbar_wait_warp(&dp_full, st & 1, &abort_flag, p.status, 1803);
        if (!ok) break;
        tc_fence_after();
        uint32_t rp[32];
        FA_TMEM_LD32_SYNC(tmem + C::kColDP + lane_off + col0, rp);
        const float* nD = &s_nD[qs][64 * h + col0];
        uint32_t dsp[16];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float4 Dd = *reinterpret_cast<const float4*>(nD + 4 * g);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 4 * g + 2 * u;
            const float2 t = add2(make_float2(__uint_as_float(rp[e]), __uint_as_float(rp[e + 1])),
                                  u ? make_float2(Dd.z, Dd.w) : make_float2(Dd.x, Dd.y));
            const float2 dsv = mul2(mul2(make_float2(pf[e], pf[e + 1]), sc2), t);
            dsp[e / 2] = pack_bf16(dsv.x, dsv.y);
          }
        }
        FA_TMEM_ST16(tmem + C::kColDP + lane_off + col0, dsp);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(&ds_ready);
      }
      if (!ok) break;
    }
    // ------------------------------------------------------------ dK, dV out
    // TMEM loads are warp-collective: every lane takes part; only rows inside
    // the sequence are stored.  `drain` completes once, after the issuer's
    // last MMA (a per-tile barrier's parity could alias an earlier phase).
    if (__all_sync(0xffffffffu, ok && !abort_flag) && it > 0)
      ok = mbar_wait_warp(&drain, 0, &abort_flag, p.status, 1807);
    const bool live = __all_sync(0xffffffffu, ok && !abort_flag);
    if (live) {
      tc_fence_after();
      const long long base_v = row_offset(p.ldv, b, hd, key) + wg * C::kDSlice;
      const long long base_k = row_offset(p.ldk, b, hd, key) + wg * C::kDSlice;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        uint32_t rr[C::kDSlice];
        const uint32_t col = (which == 0 ? C::kColDV : C::kColDK) + wg * C::kDSlice;
        if (it > 0) {
          if constexpr (C::kDSlice == 32) {
            FA_TMEM_LD32_SYNC(tmem + col + lane_off, rr);
          } else {
            FA_TMEM_LD16_SYNC(tmem + col + lane_off, rr);
          }
        } else {
#pragma unroll
          for (int e = 0; e < C::kDSlice; ++e) rr[e] = 0u;
        }
        if (key < p.N) store_row(which == 0 ? p.dv + base_v : p.dk + base_k, rr, C::kDSlice);
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
inline Bwd64Params make_dkdv64_params(const BwdArgs& a) {
  Bwd64Params p;
  p.lse = a.lse;
  p.Dvec = a.D;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.ldk = a.ldk;
  p.ldv = a.ldv;
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
  p.order = p.block_mask && a.tile_order ? a.tile_order + p.T : nullptr;  // key tiles at [T, 2T)
  return p;
}

}  // namespace
}  // namespace fa
