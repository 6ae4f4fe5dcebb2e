// Backward pass of exact attention on sm_103a tensor cores, dK and dV, with P
// recomputed on chip from Q, K and lse ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", summary page, "Key
// ideas: recomputation in the backward pass").  The gradient formulas are the
// textbook derivative of the definition (the pages do not print them): with
// S = scale Q K^T, P = exp(S - lse), D_i = rowsum(dO o O)_i,
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  dK = scale dS^T Q.
// dQ = scale dS K has a kernel of its own (one CTA per query tile, no atomics).
//
// One CTA owns a 128-key tile K_j, V_j of one (batch, head) and walks the
// query tiles Q_i that can see it (causal: i >= j; block-sparse: mask[i][j]).
// Everything is computed transposed, keys on the TMEM lanes.  TMEM columns:
//   [0, d)          dV accumulator          [d, 2d)        dK accumulator
//   [2d, 2d+128)    S^T = K_j Q_i^T, then P^T (bf16, packed two per column:
//                   warpgroup w's 32 query columns in [32w, 32w+16))
//   [2d+128, +128)  dP^T = V_j dO_i^T, then dS^T (packed the same way)
// Per query tile, with the math overlapping:
//   S^T            in two halves of 64 query columns (N = 64), both operands
//                  K-major in shared memory; half h after the previous tile's
//                  dV steps of half h, the readers of the P^T packed there
//   dP^T           after the previous dK, the last reader of dS^T (meanwhile
//                  the math computes P^T = 2^(c S^T - lse2_i) into TMEM, each
//                  half as soon as its S^T half is in)
//   dV += P^T dO_i A from TMEM, half by half as each half's P^T lands
//                  (meanwhile the math computes dS^T = scale P^T o (dP^T - D_i))
//   dK += dS^T Q_i A from TMEM
// so that a tile's S^T half waits for one half of the previous dV only.
//
// Roles (640 threads): warps 0-15 are four math warpgroups -- warpgroup w owns
// query columns [32w, 32w+32) of S^T / dP^T and d columns [w d/4, (w+1) d/4)
// of dK, dV; warp 16 is the TMA producer; warps 17, 18 and 19 issue the MMAs
// (S^T; dV, dK; dP^T).
//
// Inputs are read through 4-D TMA descriptors with their own strides; dK, dV
// are stored through theirs.  A block-sparse CTA copies its column of the tile
// mask into a shared-memory bitmap first.  The kExtra variant adds dropout
// (the keep bits of a key for 32 query rows, each Philox call drawn once by one
// of eight lanes and shared through shuffles; dV takes (P o Z)^T, dS^T the
// dropped form of dP^T, dV is scaled by 1/(1-p) at the end) and an additive bias
// (bias[query][key] added to the scaled scores before the exponential).
//
// This header holds the CTA body; the kernels that run it are in the .cu files
// (the kernel of its own and the combined backward kernel).
#pragma once
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kChunks = D / 64;
  static constexpr int kQStages = (D == 64) ? 4 : 3;   // Q ring (Q_i lives from S^T to dK)
  static constexpr int kDOStages = (D == 64) ? 4 : 2;  // dO ring
  static constexpr int kPrefetchTiles = 4;             // L2 prefetch distance (query tiles)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;
  static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;
  static constexpr int kSmem = kOffDO + kDOStages * kTileBytes + 1024;
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + 128;
  static constexpr int kMathWarps = 16;
  static constexpr int kMathThreads = kMathWarps * 32;
  static constexpr int kThreads = kMathThreads + 128;  // + producer, three MMA issuers
  static constexpr int kDSlice = D / 4;  // d columns per warpgroup in the dK / dV read-out
};

struct BwdParams {
  const float* lse;
  const float* Dvec;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  Layout ldk, ldv;
  DropParams drop;
  const float* bias;  // additive score bias or nullptr
  Layout lb;
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
struct QTileIter {
  const uint32_t* bits;
  int T, ibegin;
  __device__ int first() const { return next(ibegin); }
  __device__ int next(int i) const { return bits ? next_tile_bit(bits, i, T) : i; }
};

// n fp32 values (TMEM words) times `mult`, stored as bf16.
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t* r, int n,
                                               float mult) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  auto f = [&](int e) { return __uint_as_float(r[e]) * mult; };
  for (int g = 0; g < n / 8; ++g) {
    uint4 w;
    w.x = pack_bf16(f(8 * g), f(8 * g + 1));
    w.y = pack_bf16(f(8 * g + 2), f(8 * g + 3));
    w.z = pack_bf16(f(8 * g + 4), f(8 * g + 5));
    w.w = pack_bf16(f(8 * g + 6), f(8 * g + 7));
    d4[g] = w;
  }
}

template <int D, bool kExtra>
__device__ __forceinline__ void dkdv_cta(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                         const CUtensorMap& tmV, const CUtensorMap& tmDO, const BwdParams& p, int cta) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t kv_full, dp_ready, ds_ready, drain, drain_a, drain_c;
  // The copy of the statistics is split by warpgroup: warpgroup w reads only
  // entries [32w, 32w+32), its query columns.  stats_read[w] completes when its
  // four warps are past their last read of the tile's entries (their dS^T),
  // stats_ready[w] when its first warp has written the next tile's.
  __shared__ uint64_t stats_read[4], stats_ready[4];
  // S^T is computed and consumed in two halves of 64 query columns: half h
  // holds warpgroups 2h and 2h+1's columns, and their packed P^T.
  //   s_ready[h]: S^T half h is in TMEM (issuer A)
  //   p_ready[h]: P^T of half h is in TMEM (the 8 warps of warpgroups 2h, 2h+1)
  //   s_free[h]:  dV's K steps of half h are done, so half h may be overwritten
  //               by the next tile's S^T (issuer B)
  __shared__ uint64_t s_ready[2], p_ready[2], s_free[2];
  // q_empty[s] completes when dK of the tile in Q stage s is done (dK is the
  // last reader of Q_i: S^T was read before the math could produce dS^T): it
  // both frees the stage and tells issuer C that dS^T (in the dP^T columns) was
  // read.  do_empty[s] completes when both readers of dO_i, dV and dP^T, are
  // done: it frees the dO stage and tells issuer A that P^T (in the S^T
  // columns) was read.  Per-stage barriers keep every waiter within one phase.
  __shared__ uint64_t q_full[C::kQStages], q_empty[C::kQStages];
  __shared__ uint64_t do_full[C::kDOStages], do_empty[C::kDOStages];
  __shared__ __align__(16) float s_nl2[128];  // -lse2 of the tile's query rows
  __shared__ __align__(16) float s_nD[128];   // -D
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
  const QTileIter qtiles{p.block_mask ? mask_bits : nullptr, p.T, p.causal ? kt : 0};
  const int iend = keys_live ? p.T : 0;

  if (tid == 0) {
    mbar_init(&kv_full, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s_ready[h], 1);
      mbar_init(&p_ready[h], C::kMathWarps / 2);  // one arrival per warp of the half
      mbar_init(&s_free[h], 1);
    }
    mbar_init(&dp_ready, 1);
    mbar_init(&ds_ready, C::kMathWarps);
    for (int w = 0; w < 4; ++w) {
      mbar_init(&stats_read[w], 4);
      mbar_init(&stats_ready[w], 1);
    }
    mbar_init(&drain, 1);
    mbar_init(&drain_a, 1);
    mbar_init(&drain_c, 1);
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);  // dK, the last reader of Q_i, is done
    }
    for (int s = 0; s < C::kDOStages; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 2);  // dO_i has two readers: dV (issuer B) and dP^T (issuer C)
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
    // ------------------------------------------------------------ producer
    if (lane == 0 && iend > 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmDO);
      mbar_expect_tx(&kv_full, 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_4d(&tmK, &kv_full, smem + C::kOffK + c * C::kChunkBytes, c * 64, kt * 128, hd, b);
        tma_load_4d(&tmV, &kv_full, smem + C::kOffV + c * C::kChunkBytes, c * 64, kt * 128, hd, b);
      }
      int qcount[C::kQStages] = {}, dcount[C::kDOStages] = {};
      // L2 prefetch of the Q / dO tiles a few query tiles ahead of their loads,
      // which then find them in L2 instead of paying the DRAM latency
      int ipf = qtiles.first(), npf = 0;
      auto prefetch_upto = [&](int count) {
        for (; npf < count && ipf < iend; ++npf, ipf = qtiles.next(ipf + 1))
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
        if (!mbar_wait(&q_empty[qs], ((it / C::kQStages) & 1) ^ 1, &abort_flag, p.status, 401))
          break;
        mbar_expect_tx(&q_full[qs], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(&tmQ, &q_full[qs], smem + C::kOffQ + qs * C::kTileBytes + c * C::kChunkBytes,
                      c * 64, i * 128, hd, b);
        ++qcount[qs];
        if (!mbar_wait(&do_empty[ds], ((it / C::kDOStages) & 1) ^ 1, &abort_flag, p.status, 402))
          break;
        mbar_expect_tx(&do_full[ds], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(&tmDO, &do_full[ds],
                      smem + C::kOffDO + ds * C::kTileBytes + c * C::kChunkBytes, c * 64, i * 128, hd,
                      b);
        ++dcount[ds];
      }
      mbar_drain(&kv_full, 0);
      for (int s = 0; s < C::kQStages; ++s)
        if (qcount[s]) mbar_drain(&q_full[s], (qcount[s] - 1) & 1);
      for (int s = 0; s < C::kDOStages; ++s)
        if (dcount[s]) mbar_drain(&do_full[s], (dcount[s] - 1) & 1);
    }
  } else if (warp > C::kMathWarps) {
    // ------------------------------------------------------------ MMA issuers
    // Three issuing threads, so that a wait on one dependency chain never holds
    // back another's MMAs (an MMA costs its issuing thread about as long as the
    // tensor core takes to run it):
    //   A (warp 17): S^T  -- gated by Q_i and by the previous tile's dV (the
    //                reader of the S^T columns, where P^T sits)
    //   B (warp 18): dV and dK -- gated by the math (P^T, dS^T)
    //   C (warp 19): dP^T -- gated by dO_i and by the previous tile's dK (the
    //                reader of the dP^T columns, where dS^T sits)
    const int role = warp - C::kMathWarps - 1;  // 0: A, 1: B, 2: C
    const bool issuer_a = role == 0, issuer_c = role == 2;
    if (lane == 0 && iend > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);   // dP^T
      constexpr uint32_t idesc_s64 = idesc_bf16(128, 64, false, false);  // S^T halves
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, false, true);   // dV, dK
      const uint32_t sK = smem_addr(smem + C::kOffK), sV = smem_addr(smem + C::kOffV);
      const uint32_t sQ0 = smem_addr(smem + C::kOffQ), sDO0 = smem_addr(smem + C::kOffDO);
      // operand descriptors: built once per buffer; an operand's K step adds
      // its byte offset >> 4 to the start-address field (every buffer lies
      // below 256 KB, so the 14-bit field never carries)
      const uint64_t dK_k = sdesc_sw128(sK, 16, 1024), dV_k = sdesc_sw128(sV, 16, 1024);
      bool ok = role == 1 || mbar_wait(&kv_full, 0, &abort_flag, p.status, 501);  // K, V
      int it = 0;
      for (int i = qtiles.first(); ok && i < iend; i = qtiles.next(i + 1), ++it) {
        const int qs = it % C::kQStages, ds = it % C::kDOStages;
        const uint32_t sQ = sQ0 + qs * C::kTileBytes, sDO = sDO0 + ds * C::kTileBytes;
        if (!issuer_c) {  // A and B read Q_i
          ok = mbar_wait(&q_full[qs], (it / C::kQStages) & 1, &abort_flag, p.status, 502);
          if (!ok) break;
        }
        if (issuer_a) {
          const uint64_t dQ_k = sdesc_sw128(sQ, 16, 1024);
          for (int h = 0; h < 2 && ok; ++h) {
            // P^T of the previous tile's half h sits in those S^T columns until
            // dV has read it
            if (it > 0) ok = mbar_wait(&s_free[h], (it - 1) & 1, &abort_flag, p.status, 503);
            if (!ok) break;
            tc_fence_after();
            // S^T half h = K Q^T of query rows [64h, 64h + 64): N = 64; those
            // rows start 64 x 128 bytes into each chunk of the Q tile
            const uint64_t dQh = dQ_k + ((uint32_t)(64 * 128 * h) >> 4);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t koff = ((ks >> 2) * C::kChunkBytes + (ks & 3) * 32) >> 4;
              mma_ss(tmem + C::kColS + 64 * h, dK_k + koff, dQh + koff, idesc_s64, ks > 0);
            }
            mma_commit(&s_ready[h]);
          }
          if (!ok) break;
        } else if (issuer_c) {
          const uint64_t dDO_k = sdesc_sw128(sDO, 16, 1024);
          // dS^T of the previous tile sits in the dP^T columns until its dK is done
          if (it > 0)
            ok = mbar_wait(&q_empty[(it - 1) % C::kQStages], ((it - 1) / C::kQStages) & 1,
                           &abort_flag, p.status, 504);
          if (ok) ok = mbar_wait(&do_full[ds], (it / C::kDOStages) & 1, &abort_flag, p.status, 506);
          if (!ok) break;
          tc_fence_after();
          // dP^T = V dO^T
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t koff = ((ks >> 2) * C::kChunkBytes + (ks & 3) * 32) >> 4;
            mma_ss(tmem + C::kColDP, dV_k + koff, dDO_k + koff, idesc_s, ks > 0);
          }
          mma_commit(&dp_ready);
          mma_commit(&do_empty[ds]);  // this reader of dO_i is done
        } else {
          const uint64_t dQ_mn = sdesc_sw128(sQ, C::kChunkBytes, 1024);
          const uint64_t dDO_mn = sdesc_sw128(sDO, C::kChunkBytes, 1024);
          const uint32_t acc = it > 0 ? 1u : 0u;
          ok = mbar_wait(&do_full[ds], (it / C::kDOStages) & 1, &abort_flag, p.status, 508);
          // dV += P^T dO, half by half as each half's P^T lands (P^T in TMEM:
          // warpgroup w's 32 query columns sit packed in columns [32w, 32w+16)
          // of the S^T region; half h = K steps 4h .. 4h + 3)
          for (int h = 0; h < 2 && ok; ++h) {
            ok = mbar_wait(&p_ready[h], it & 1, &abort_flag, p.status, 505);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int ks = 4 * h + k4;
              mma_ts(tmem + C::kColDV, tmem + C::kColS + 32 * (ks >> 1) + 8 * (ks & 1),
                     dDO_mn + ks * (2048 >> 4), idesc_acc, acc | (ks > 0));
            }
            mma_commit(&s_free[h]);
          }
          if (!ok) break;
          mma_commit(&do_empty[ds]);  // this reader of dO_i is done
          ok = mbar_wait(&ds_ready, it & 1, &abort_flag, p.status, 507);
          if (!ok) break;
          tc_fence_after();
          // dK += dS^T Q (dS^T in TMEM: warpgroup w's columns packed in
          // [32w, 32w+16) of the dP^T region)
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ts(tmem + C::kColDK, tmem + C::kColDP + 32 * (ks >> 1) + 8 * (ks & 1),
                   dQ_mn + ks * (2048 >> 4), idesc_acc, acc | (ks > 0));
          mma_commit(&q_empty[qs]);
        }
      }
      // each issuer's MMAs are complete once its drain barrier flips; B's last
      // MMA (dK) follows every MMA of A and C (B's last dV waited for the last
      // S^T halves through p_ready, its last dK for the last dP^T through ds_ready),
      // so `drain` alone tells the math that all are done
      uint64_t* my_drain = issuer_a ? &drain_a : issuer_c ? &drain_c : &drain;
      mma_commit(my_drain);
      mbar_drain(my_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ math warpgroups
    const int wg = warp >> 2;               // 0..3
    const int tq = tid & 127;               // TMEM lane: key row (S^T) / query row (dQ)
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int key = kt * 128 + tq;
    const bool key_live = key < kv_limit;
    const size_t head_row0 = (size_t)bh * p.N;
    const int col0 = wg * 32;               // this warpgroup's query columns
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    const float2 sc2 = make_float2(p.scale, p.scale);
    const bool bias_on = kExtra && p.bias != nullptr;
    int it = 0;
    bool ok = true;
    // Statistics of one query row: loaded raw (lse, D) by a lane of the
    // warpgroup's first warp (lane l: query column col0 + l), converted to
    // what the math uses (-lse2, -D) only when stored, so that the load's
    // latency is not waited for before then.
    const bool stats_writer = (warp & 3) == 0;
    struct RowStats {
      float nl2, nd;
    };
    auto load_stats = [&](int qt) {
      RowStats st{-INFINITY, 0.f};  // rows past the end: P = 0
      const int q = qt * 128 + col0 + lane;
      if (qt < iend && q < p.N) {
        st.nl2 = p.lse[head_row0 + q];
        st.nd = p.Dvec[head_row0 + q];
      }
      return st;
    };
    auto finish_stats = [](RowStats st) {
      asm volatile("" : "+f"(st.nl2), "+f"(st.nd));  // first use of the loaded values
      // rows with no visible key (lse = -inf) keep -lse2 = -inf: P = 0
      st.nl2 = st.nl2 == -INFINITY ? -INFINITY : -st.nl2 * kLog2e;
      st.nd = -st.nd;
      return st;
    };
    // dropout: the first tile's keep bits (every math lane takes part: shuffles)
    uint32_t keep_next = ~0u;
    if (kExtra && p.drop.t && iend > 0)
      keep_next = keep_bits_of_key(p.drop, (uint32_t)bh, key, qtiles.first() * 128 + col0);
    if (stats_writer && iend > 0) {
      const RowStats st = finish_stats(load_stats(qtiles.first()));
      s_nl2[col0 + lane] = st.nl2;
      s_nD[col0 + lane] = st.nd;
      mbar_arrive_warp(&stats_ready[wg]);
    }
    for (int i = qtiles.first(); i < iend; i = qtiles.next(i + 1), ++it) {
      // ---- the next tile's statistics: loaded now, stored once the
      // warpgroup's threads are past this tile's dS (the loads' latency hides
      // behind the MMAs)
      RowStats next_st{};
      if (stats_writer) next_st = load_stats(qtiles.next(i + 1));
      // dropout: keep bits of this key for the warpgroup's 32 query rows (all
      // set without dropout), drawn during the previous tile; bias:
      // bias[query][key] times log2(e) of those rows, in pf, read while S^T is
      // computed
      const uint32_t keep = kExtra ? keep_next : 0u;
      float pf[32];
      if (kExtra && bias_on) {
        const int qr0 = i * 128 + col0;
        const float* bcol = p.bias + row_offset(p.lb, b, hd, qr0) + key;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          pf[c] = (key < p.N && qr0 + c < p.N) ? __ldg(bcol + (long long)c * p.lb.n) * kLog2e : 0.f;
      }
      ok = mbar_wait_warp(&stats_ready[wg], it & 1, &abort_flag, p.status, 601);
      if (ok) ok = mbar_wait_warp(&s_ready[wg >> 1], it & 1, &abort_flag, p.status, 602);
      if (!ok) break;
      tc_fence_after();
      const int q0 = i * 128;
      const bool masked = !key_live || (p.causal && key > q0 + col0);
      // ---- P^T for the warpgroup's 32 columns (while dP^T is computed); packed
      // P^T of half h goes over S^T columns [col0 + 8h, col0 + 8h + 8), which
      // were read in half 0
      uint32_t rs_all[32];
      FA_TMEM_LD32_SYNC(tmem + C::kColS + lane_off + col0, rs_all);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c0 = col0 + 16 * h;
        const uint32_t* rs = rs_all + 16 * h;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float4 L = *reinterpret_cast<const float4*>(&s_nl2[c0 + 4 * g]);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 4 * g + 2 * u;
            float2 x = fma2(make_float2(__uint_as_float(rs[e]), __uint_as_float(rs[e + 1])), c2,
                            u ? make_float2(L.z, L.w) : make_float2(L.x, L.y));
            if (kExtra && bias_on) x = add2(x, make_float2(pf[16 * h + e], pf[16 * h + e + 1]));
            pf[16 * h + e] = ex2(x.x);
            pf[16 * h + e + 1] = ex2(x.y);
          }
        }
        if (masked) {  // causal diagonal tiles and padded keys
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (!key_live || key > q0 + c0 + e) pf[16 * h + e] = 0.f;
        }
        uint32_t pp[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          float a0 = pf[16 * h + e], a1 = pf[16 * h + e + 1];
          if constexpr (kExtra) {  // dV takes (P o Z)^T; the 1 / (1 - p) is applied at the end
            if (!((keep >> (16 * h + e)) & 1u)) a0 = 0.f;
            if (!((keep >> (16 * h + e + 1)) & 1u)) a1 = 0.f;
          }
          pp[e / 2] = pack_bf16(a0, a1);
        }
        FA_TMEM_ST8(tmem + C::kColS + lane_off + col0 + 8 * h, pp);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&p_ready[wg >> 1]);
      // dropout: the next tile's keep bits, drawn while dP^T is computed
      if (kExtra && p.drop.t) {
        const int inext = qtiles.next(i + 1);
        keep_next = inext < iend
                        ? keep_bits_of_key(p.drop, (uint32_t)bh, key, inext * 128 + col0)
                        : ~0u;
      }
      // ---- dS^T = scale P^T o (dP^T - D) (while dV is computed): packed bf16
      // over dP^T columns [col0, col0 + 16), which this thread has read
      ok = mbar_wait_warp(&dp_ready, it & 1, &abort_flag, p.status, 608);
      if (!ok) break;
      tc_fence_after();
      uint32_t dsp[16];
      uint32_t rp_all[32];
      FA_TMEM_LD32_SYNC(tmem + C::kColDP + lane_off + col0, rp_all);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c0 = col0 + 16 * h;
        const uint32_t* rp = rp_all + 16 * h;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float4 Dd = *reinterpret_cast<const float4*>(&s_nD[c0 + 4 * g]);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 4 * g + 2 * u;
            const float2 dpv = make_float2(__uint_as_float(rp[e]), __uint_as_float(rp[e + 1]));
            const float2 nD = u ? make_float2(Dd.z, Dd.w) : make_float2(Dd.x, Dd.y);
            float2 t;
            if constexpr (kExtra) {
              // dS^T = P^T o (Z o dP^T / (1 - p) - D): dropped entries keep only -D
              const int c = 16 * h + e;
              const float2 zr = make_float2(((keep >> c) & 1u) ? p.drop.rp : 0.f,
                                            ((keep >> (c + 1)) & 1u) ? p.drop.rp : 0.f);
              t = fma2(dpv, zr, nD);
            } else {
              t = add2(dpv, nD);
            }
            const float2 dsv = mul2(mul2(make_float2(pf[16 * h + e], pf[16 * h + e + 1]), sc2), t);
            dsp[8 * h + e / 2] = pack_bf16(dsv.x, dsv.y);
          }
        }
      }
      FA_TMEM_ST16(tmem + C::kColDP + lane_off + col0, dsp);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&ds_ready);
      mbar_arrive_warp(&stats_read[wg]);
      // ---- the next tile's statistics replace this tile's once the
      // warpgroup's four warps are past their last read of them
      if (stats_writer) {
        if (!mbar_wait_warp(&stats_read[wg], it & 1, &abort_flag, p.status, 600)) break;
        const RowStats st = finish_stats(next_st);
        s_nl2[col0 + lane] = st.nl2;
        s_nD[col0 + lane] = st.nd;
        mbar_arrive_warp(&stats_ready[wg]);
      }
    }
    // ------------------------------------------------------------ dK, dV out
    // TMEM loads are warp-collective: every lane takes part; only rows inside
    // the sequence are stored.  `drain` completes once, after the issuer's
    // last MMA (a per-tile barrier's parity could alias an earlier phase).
    if (__all_sync(0xffffffffu, ok && !abort_flag) && it > 0)
      ok = mbar_wait_warp(&drain, 0, &abort_flag, p.status, 607);
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
        if (key < p.N)
          store_row_bf16(which == 0 ? p.dv + base_v : p.dk + base_k, rr, C::kDSlice,
                         (kExtra && which == 0) ? p.drop.rp : 1.f);
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
inline BwdParams make_dkdv_params(const BwdArgs& a) {
  BwdParams p;
  p.lse = a.lse;
  p.Dvec = a.D;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.ldk = a.ldk;
  p.ldv = a.ldv;
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
  p.order = p.block_mask && a.tile_order ? a.tile_order + p.T : nullptr;  // key tiles at [T, 2T)
  return p;
}

}  // namespace
}  // namespace fa
