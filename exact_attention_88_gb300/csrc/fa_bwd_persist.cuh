// Backward pass of exact attention, dQ, with persistent CTAs: one CTA per SM
// takes query tiles (units) one after another instead of one CTA per unit, so
// that a unit's first loads and MMAs run under the previous unit's last key
// tile and its epilogue.  (A trace of the one-CTA-per-unit dQ kernel on a
// 16K-token causal call put a fixed 5.3 us per CTA, plus 0.6 us between CTAs,
// against 1.07 us per key tile; taken persistently, 2.8 us per unit.)
//
// The arithmetic is that of the dQ CTA (fa_bwd_dq.cuh; "FlashAttention: Fast
// and Memory-Efficient Exact Attention with IO-Awareness", summary page, "Key
// ideas: recomputation in the backward pass"), with the same TMEM columns,
// rings and roles, and dQ is bit-identical to the one-per-unit CTA's: a unit
// runs the same MMAs in the same order.  The combined backward kernel uses
// it for the calls without a block mask, key padding, dropout or a bias at
// d = 128.
//
// Units: the combined kernel's dK/dV CTAs take units [0, n0); [n0, n) are the
// dQ query tiles in their grid order (heaviest first).  The persistent CTA x
// (x >= n0) starts with unit x; its producer takes every later unit from a
// counter in the workspace (zeroed by the preprocess before the kernel),
// gridDim + the counter's old value, and hands it to the other roles through
// a ring of shared-memory slots.  Units go out in index order to whichever CTA
// asks first, as the hardware would dispatch one CTA per unit, so the load
// balance is that of the grid order.
//
// Across units:
//   - Q_i, dO_i have one buffer: the producer loads the next unit's once the
//     unit's last S and dP (their readers) are done (qd_empty: one commit
//     from each of the two issuers), after an L2 prefetch issued when it took
//     the unit;
//   - the dQ accumulator is read out by the math warps once the unit's last
//     dQ MMA is done (acc_ready), which then arrive on acc_free; the next
//     unit's first dQ MMA waits for that;
//   - every per-tile barrier and ring keeps counting across units, so the
//     next unit's first S needs only the math to have read the previous S.
// (The same treatment of the dK/dV CTA ran its query tiles 7.5 % slower,
// 1.75 against 1.62 us a tile on the same box, even one unit per CTA, which
// ate its 3.7 us per unit of savings; that CTA is kept one per unit.)
#pragma once
#include "fa_bwd_dq.cuh"

namespace fa {
namespace {

constexpr int kUnitRing = 4;
// One arrival each from the three MMA issuers and from each of the 16 math warps.
constexpr int kUnitConsumers = 3 + 16;

// Shared-memory slots through which the producer hands units to the others.
struct UnitRing {
  int id[kUnitRing];
  uint64_t full[kUnitRing], empty[kUnitRing];
};

__device__ __forceinline__ void unit_ring_init(UnitRing& r) {
  for (int s = 0; s < kUnitRing; ++s) {
    mbar_init(&r.full[s], 1);
    mbar_init(&r.empty[s], kUnitConsumers);
  }
}

// The k-th unit after a body's first (k >= 1) goes to slot (k - 1) % R; the
// slot's previous unit must have been read by every consumer.
__device__ __forceinline__ bool unit_publish(UnitRing& r, int k, int id, int* abort_flag,
                                             int* status, int site) {
  const int s = (k - 1) % kUnitRing, use = (k - 1) / kUnitRing;
  if (use > 0 && !mbar_wait(&r.empty[s], (use - 1) & 1, abort_flag, status, site)) return false;
  r.id[s] = id;
  mbar_arrive(&r.full[s]);  // release: the id is visible to whoever sees the phase
  return true;
}

// The k-th unit (k >= 1), for one consumer thread; returns `done` when the
// wait gave up.
__device__ __forceinline__ int unit_take(UnitRing& r, int k, int done, int* abort_flag,
                                         int* status, int site) {
  const int s = (k - 1) % kUnitRing, use = (k - 1) / kUnitRing;
  if (!mbar_wait(&r.full[s], use & 1, abort_flag, status, site)) return done;
  const int id = *reinterpret_cast<volatile int*>(&r.id[s]);
  mbar_arrive(&r.empty[s]);
  return id;
}

// The same for a whole warp (lane 0 waits and arrives; the id is broadcast).
__device__ __forceinline__ int unit_take_warp(UnitRing& r, int k, int done, int* abort_flag,
                                              int* status, int site) {
  int id = done;
  if ((threadIdx.x & 31) == 0) id = unit_take(r, k, done, abort_flag, status, site);
  return __shfl_sync(0xffffffffu, id, 0);
}

// The next unit from the counter.
__device__ __forceinline__ int unit_fetch(int* counter) {
  return (int)gridDim.x + atomicAdd(counter, 1);
}

// ---------------------------------------------------------------------------
// dQ units
// ---------------------------------------------------------------------------
struct QueryUnit {
  int qi, bh, b, hd, jend;  // query tile, (batch, head), key tiles [0, jend)
};

__device__ __forceinline__ QueryUnit query_unit(const DqParams& p, int v) {
  QueryUnit u;
  int order;
  grid_order(v, p.BH, p.T, p.group, &order, &u.bh);
  u.qi = p.T - 1 - order;
  u.b = u.bh / p.H;
  u.hd = u.bh - u.b * p.H;
  u.jend = p.causal ? u.qi + 1 : p.T;
  return u;
}

// Runs the dQ units of this CTA from `first` (a unit in [n0, n)) to the end of
// the queue.
template <int D>
__device__ __forceinline__ void dq_persist(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                           const CUtensorMap& tmV, const CUtensorMap& tmDO,
                                           const DqParams& p, uint32_t tmem, int first, int n0,
                                           int n, int* counter) {
  using C = DqCfg<D>;
  static_assert(kUnitConsumers == 3 + C::kMathWarps,
                "every MMA issuer and every math warp takes each unit from the ring");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t qd_full, qd_empty, acc_ready, acc_free, s_full, s_free;
  __shared__ uint64_t drain_s, drain_p, drain_q;
  __shared__ uint64_t ds_ready[2];
  __shared__ uint64_t k_full[C::kKStages], dq_done[C::kKStages];
  __shared__ uint64_t v_full[C::kVStages], dp_full[C::kVStages];
  __shared__ UnitRing ring;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&qd_full, 1);
    mbar_init(&qd_empty, 2);  // the unit's last S and last dP
    mbar_init(&acc_ready, 1);
    mbar_init(&acc_free, C::kMathWarps);
    mbar_init(&s_full, 1);
    mbar_init(&s_free, C::kMathWarps);
    mbar_init(&drain_s, 1);
    mbar_init(&drain_p, 1);
    mbar_init(&drain_q, 1);
    for (int x = 0; x < 2; ++x) mbar_init(&ds_ready[x], C::kMathWarps);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&dq_done[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&dp_full[s], 1);
    }
    unit_ring_init(ring);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == C::kMathWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int kcount[C::kKStages] = {}, vcount[C::kVStages] = {}, qdcount = 0;
      int unit = first, k = 0, u = 0;
      bool ok = true;
      while (ok && unit < n) {
        const QueryUnit U = query_unit(p, unit - n0);
        if (k > 0) ok = mbar_wait(&qd_empty, (k - 1) & 1, &abort_flag, p.status, 1701);
        if (!ok) break;
        ++qdcount;
        mbar_expect_tx(&qd_full, 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_4d(&tmQ, &qd_full, smem + C::kOffQ + c * C::kChunkBytes, c * 64, U.qi * 128,
                      U.hd, U.b);
          tma_load_4d(&tmDO, &qd_full, smem + C::kOffDO + c * C::kChunkBytes, c * 64, U.qi * 128,
                      U.hd, U.b);
        }
        int jpf = 0;
        auto prefetch_upto = [&](int last) {
          for (; jpf < min(last, U.jend); ++jpf)
            for (int c = 0; c < C::kChunks; ++c) {
              tma_prefetch_4d(&tmK, c * 64, jpf * 128, U.hd, U.b);
              tma_prefetch_4d(&tmV, c * 64, jpf * 128, U.hd, U.b);
            }
        };
        prefetch_upto(C::kPrefetchTiles);
        for (int j = 0; j < U.jend; ++j, ++u) {
          prefetch_upto(j + 1 + C::kPrefetchTiles);
          const int ks = u % C::kKStages, vs = u % C::kVStages;
          ok = mbar_wait(&dq_done[ks], ((u / C::kKStages) & 1) ^ 1, &abort_flag, p.status, 1702);
          if (!ok) break;
          mbar_expect_tx(&k_full[ks], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(&tmK, &k_full[ks], smem + C::kOffK + ks * C::kTileBytes + c * C::kChunkBytes,
                        c * 64, j * 128, U.hd, U.b);
          ++kcount[ks];
          ok = mbar_wait(&dp_full[vs], ((u / C::kVStages) & 1) ^ 1, &abort_flag, p.status, 1703);
          if (!ok) break;
          mbar_expect_tx(&v_full[vs], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(&tmV, &v_full[vs], smem + C::kOffV + vs * C::kTileBytes + c * C::kChunkBytes,
                        c * 64, j * 128, U.hd, U.b);
          ++vcount[vs];
        }
        if (!ok) break;
        const int next = unit_fetch(counter);
        if (next < n) {
          const QueryUnit V = query_unit(p, next - n0);
          for (int c = 0; c < C::kChunks; ++c) {
            tma_prefetch_4d(&tmQ, c * 64, V.qi * 128, V.hd, V.b);
            tma_prefetch_4d(&tmDO, c * 64, V.qi * 128, V.hd, V.b);
          }
        }
        ok = unit_publish(ring, k + 1, next, &abort_flag, p.status, 1704);
        unit = next;
        ++k;
      }
      if (!ok) abort_flag = 1;
      if (qdcount > 0) mbar_drain(&qd_full, (qdcount - 1) & 1);
      for (int s = 0; s < C::kKStages; ++s)
        if (kcount[s]) mbar_drain(&k_full[s], (kcount[s] - 1) & 1);
      for (int s = 0; s < C::kVStages; ++s)
        if (vcount[s]) mbar_drain(&v_full[s], (vcount[s] - 1) & 1);
    }
  } else if (warp > C::kMathWarps) {
    // ------------------------------------------------------------ MMA issuers
    //   warp 17: S, warp 18: dP, warp 19: dQ
    const int role = warp - (C::kMathWarps + 1);
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_dq = idesc_bf16(128, D, false, true);
      const uint64_t dQ_k = sdesc_sw128(smem_addr(smem + C::kOffQ), 16, 1024);
      const uint64_t dDO_k = sdesc_sw128(smem_addr(smem + C::kOffDO), 16, 1024);
      const uint32_t sK = smem_addr(smem + C::kOffK), sV = smem_addr(smem + C::kOffV);
      int unit = first, k = 0, u = 0;
      bool ok = true;
      while (ok && unit < n) {
        const QueryUnit U = query_unit(p, unit - n0);
        if (role != 2) ok = mbar_wait(&qd_full, k & 1, &abort_flag, p.status, 1800);
        for (int j = 0, lu = 0; ok && j < U.jend; ++j, ++lu, ++u) {
          if (role == 0) {
            const int ks = u % C::kKStages;
            if (u > 0) ok = mbar_wait(&s_free, (u - 1) & 1, &abort_flag, p.status, 1801);
            if (ok) ok = mbar_wait(&k_full[ks], (u / C::kKStages) & 1, &abort_flag, p.status, 1802);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dK_k = sdesc_sw128(sK + ks * C::kTileBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
              mma_ss(tmem + C::kColS, dQ_k + off, dK_k + off, idesc_s, kk > 0);
            }
            mma_commit(&s_full);
          } else if (role == 1) {
            const int vs = u % C::kVStages;
            if (u >= 2)
              ok = mbar_wait(&dq_done[(u - 2) % C::kKStages], ((u - 2) / C::kKStages) & 1,
                             &abort_flag, p.status, 1803);
            if (ok) ok = mbar_wait(&v_full[vs], (u / C::kVStages) & 1, &abort_flag, p.status, 1804);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dV_k = sdesc_sw128(sV + vs * C::kTileBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
              mma_ss(tmem + C::kColDP + 128 * vs, dDO_k + off, dV_k + off, idesc_s, kk > 0);
            }
            mma_commit(&dp_full[vs]);
          } else {
            const int ks = u % C::kKStages;
            ok = mbar_wait(&k_full[ks], (u / C::kKStages) & 1, &abort_flag, p.status, 1805);
            if (ok) ok = mbar_wait(&ds_ready[u & 1], (u >> 1) & 1, &abort_flag, p.status, 1806);
            // the previous unit's dQ must have been read out by every math
            // warp before this unit's first MMA overwrites it
            if (ok && lu == 0 && k > 0)
              ok = mbar_wait(&acc_free, (k - 1) & 1, &abort_flag, p.status, 1807);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dK_mn = sdesc_sw128(sK + ks * C::kTileBytes, C::kChunkBytes, 1024);
            const uint32_t tA = tmem + C::kColDP + 128 * (u & 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C::kColDQ, tA + 32 * (kk >> 1) + 8 * (kk & 1),
                     dK_mn + kk * (2048 >> 4), idesc_dq, (lu > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&dq_done[ks]);
          }
        }
        if (!ok) break;
        // S and dP: the last readers of Q, dO; dQ: the unit's accumulator is complete
        mma_commit(role == 2 ? &acc_ready : &qd_empty);
        unit = unit_take(ring, k + 1, n, &abort_flag, p.status, 1810 + role);
        ++k;
      }
      if (!ok) abort_flag = 1;
      uint64_t* my_drain = role == 0 ? &drain_s : role == 1 ? &drain_p : &drain_q;
      mma_commit(my_drain);
      mbar_drain(my_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ math warpgroups
    const int wg = warp >> 2;
    const int tq = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int col0 = wg * 32;
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    const float2 sc2 = make_float2(p.scale, p.scale);
    // this row's raw lse and D in unit U
    auto row_stats = [&](const QueryUnit& U, float* l, float* dd) {
      const int q = U.qi * 128 + tq;
      *l = -INFINITY;
      *dd = 0.f;
      if (q < p.N) {
        *l = p.lse[(size_t)U.bh * p.N + q];
        *dd = p.Dvec[(size_t)U.bh * p.N + q];
      }
    };
    int unit = first, k = 0, u = 0;
    bool ok = true;
    float l_raw = -INFINITY, d_raw = 0.f;
    if (unit < n) row_stats(query_unit(p, unit - n0), &l_raw, &d_raw);
    while (unit < n) {
      const QueryUnit U = query_unit(p, unit - n0);
      const int q = U.qi * 128 + tq;
      const float nl2 = l_raw == -INFINITY ? -INFINITY : -l_raw * kLog2e;
      const float2 nl22 = make_float2(nl2, nl2), nd2 = make_float2(-d_raw, -d_raw);
      int next = n;
      for (int j = 0; j < U.jend; ++j, ++u) {
        const int x = u & 1;
        const uint32_t tS = tmem + C::kColS + lane_off + col0;
        const uint32_t tP = tmem + C::kColDP + 128 * x + lane_off + col0;
        const int key0 = j * 128 + col0;
        if (j + 1 == U.jend) {  // the next unit and its row statistics, early
          next = unit_take_warp(ring, k + 1, n, &abort_flag, p.status, 1901);
          if (next < n) row_stats(query_unit(p, next - n0), &l_raw, &d_raw);
        }
        ok = mbar_wait_warp(&s_full, u & 1, &abort_flag, p.status, 1902);
        if (!ok) break;
        tc_fence_after();
        int lim = p.N - key0;
        if (p.causal) lim = min(lim, q - key0 + 1);
        float pf[32];
        uint32_t rs_all[32];
        FA_TMEM_LD32_SYNC(tS, rs_all);
        tc_fence_before();
        mbar_arrive_warp(&s_free);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 t =
              fma2(make_float2(__uint_as_float(rs_all[e]), __uint_as_float(rs_all[e + 1])), c2, nl22);
          pf[e] = ex2(t.x);
          pf[e + 1] = ex2(t.y);
        }
        if (lim < 32) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e >= lim) pf[e] = 0.f;
        }
        ok = mbar_wait_warp(&dp_full[x], (u >> 1) & 1, &abort_flag, p.status, 1903);
        if (!ok) break;
        tc_fence_after();
        uint32_t dsp[16];
        uint32_t rp_all[32];
        FA_TMEM_LD32_SYNC(tP, rp_all);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 dpv = make_float2(__uint_as_float(rp_all[e]), __uint_as_float(rp_all[e + 1]));
          const float2 dsv = mul2(mul2(make_float2(pf[e], pf[e + 1]), sc2), add2(dpv, nd2));
          dsp[e / 2] = pack_bf16(dsv.x, dsv.y);
        }
        FA_TMEM_ST16(tP, dsp);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(&ds_ready[x]);
      }
      if (!__all_sync(0xffffffffu, ok && !abort_flag)) break;
      // ---- dQ of the unit out, then the columns are free for the next
      ok = mbar_wait_warp(&acc_ready, k & 1, &abort_flag, p.status, 1904);
      if (!ok) break;
      tc_fence_after();
      uint32_t r[C::kDSlice];
      if constexpr (C::kDSlice == 32) {
        FA_TMEM_LD32_SYNC(tmem + C::kColDQ + lane_off + wg * C::kDSlice, r);
      } else {
        FA_TMEM_LD16_SYNC(tmem + C::kColDQ + lane_off + wg * C::kDSlice, r);
      }
      tc_fence_before();
      mbar_arrive_warp(&acc_free);
      if (q < p.N) {
        uint4* dst = reinterpret_cast<uint4*>(p.dq + row_offset(p.ldq, U.b, U.hd, q) + wg * C::kDSlice);
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
      unit = next;
      ++k;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

}  // namespace
}  // namespace fa
