// Backward pass of exact attention on sm_103a tensor cores: dK, dV and the
// dQ contributions, with P recomputed on chip from Q, K and lse ("FlashAttention:
// Fast and Memory-Efficient Exact Attention with IO-Awareness", summary page,
// "Key ideas: recomputation in the backward pass").  The gradient formulas
// are the textbook derivative of the definition (the pages do not print
// them): with S = scale Q K^T, P = exp(S - lse), D_i = rowsum(dO o O)_i,
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),
//   dK = scale dS^T Q,  dQ = scale dS K.
//
// One CTA owns a 128-key tile K_j, V_j of one (batch, head) and walks the
// query tiles Q_i that can see it (causal: i >= j; block-sparse: mask[i][j]).
// Everything is computed transposed, keys on the TMEM lanes:
//   S^T  = K_j Q_i^T      -> TMEM [0,128)        (tcgen05, both K-major)
//   dP^T = V_j dO_i^T     -> TMEM [128,256)
//   P^T  = 2^(c S^T - lse2_i),  dS^T = scale P^T o (dP^T - D_i)    (warps 0-3,
//          one key row per thread, written as bf16 to swizzled shared memory)
//   dV  += P^T dO_i       -> TMEM [256, 256+d)   (B operand MN-major)
//   dK  += dS^T Q_i       -> TMEM [256+d, 256+2d)
//   dQ_i = dS K_j         -> TMEM [0, d), the same shared-memory dS^T tile
//          read through an MN-major descriptor; warps 0-3 add it into the
//          fp32 dq accumulator with vector reductions.
// Roles: warps 0-3 compute, warp 4 TMA producer, warp 5 MMA issuer.
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kChunks = D / 64;
  static constexpr int kSBytes = 128 * 128 * 2;  // P^T or dS^T tile, bf16
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;
  static constexpr int kOffDO = kOffQ + kTileBytes;
  static constexpr int kOffP = kOffDO + kTileBytes;
  static constexpr int kOffDS = kOffP + kSBytes;
  static constexpr int kSmem = kOffDS + kSBytes + 1024;
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D, kColDQ = 0;
};

struct BwdParams {
  const float* lse;
  const float* Dvec;
  float* dq_acc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  int H, N, T, BH;
  float scale, scale_log2;
  int causal;
  int* status;
};

// Query tiles i that see key tile kt: i in [ibegin, T), block-mask column kt.
struct QTileIter {
  const uint8_t* mask;  // block mask base or nullptr
  int T, kt, ibegin;
  __device__ int first() const { return next(ibegin); }
  __device__ int next(int i) const {
    if (mask)
      while (i < T && mask[(size_t)i * T + kt] == 0) ++i;
    return i;
  }
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t kv_full, qdo_full, qdo_empty, s_full, p_full, mma_done, dq_free, drain;
  __shared__ uint64_t stats_ready[2];  // lse/D of a query tile staged (128 arrivals)
  __shared__ float s_lse2[2][128], s_D[2][128];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lin = blockIdx.x;
  const int kt = lin / p.BH;  // key tile (causal: low tiles have the most work: first)
  const int bh = lin % p.BH;
  const int b = bh / p.H;
  int kv_limit = p.N;
  if (p.kv_len) kv_limit = max(0, min(p.kv_len[b], p.N));
  const bool keys_live = kt * 128 < kv_limit;  // else every key of the tile is padding
  const QTileIter qtiles{p.block_mask, p.T, kt, p.causal ? kt : 0};
  const int iend = keys_live ? p.T : 0;

  if (tid == 0) {
    mbar_init(&kv_full, 1);
    mbar_init(&qdo_full, 1);
    mbar_init(&qdo_empty, 1);
    mbar_init(&s_full, 1);
    mbar_init(&p_full, 128);
    mbar_init(&mma_done, 1);
    mbar_init(&dq_free, 128);
    mbar_init(&drain, 1);
    mbar_init(&stats_ready[0], 128);
    mbar_init(&stats_ready[1], 128);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(&tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && iend > 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmDO);
      mbar_expect_tx(&kv_full, 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(&tmK, &kv_full, smem + C::kOffK + c * C::kChunkBytes, c * 64, kt * 128, bh);
        tma_load_3d(&tmV, &kv_full, smem + C::kOffV + c * C::kChunkBytes, c * 64, kt * 128, bh);
      }
      int it = 0;
      for (int i = qtiles.first(); i < iend; i = qtiles.next(i + 1), ++it) {
        if (!mbar_wait(&qdo_empty, (it & 1) ^ 1, &abort_flag, p.status, 401)) break;
        mbar_expect_tx(&qdo_full, 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(&tmQ, &qdo_full, smem + C::kOffQ + c * C::kChunkBytes, c * 64, i * 128, bh);
          tma_load_3d(&tmDO, &qdo_full, smem + C::kOffDO + c * C::kChunkBytes, c * 64, i * 128, bh);
        }
      }
      mbar_drain(&kv_full, 0);
      if (it > 0) mbar_drain(&qdo_full, (it - 1) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && iend > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, false, true);   // dV, dK
      constexpr uint32_t idesc_dq = idesc_bf16(128, D, true, true);     // dQ
      const uint32_t sK = smem_addr(smem + C::kOffK), sV = smem_addr(smem + C::kOffV);
      const uint32_t sQ = smem_addr(smem + C::kOffQ), sDO = smem_addr(smem + C::kOffDO);
      const uint32_t sP = smem_addr(smem + C::kOffP), sDS = smem_addr(smem + C::kOffDS);
      bool ok = mbar_wait(&kv_full, 0, &abort_flag, p.status, 501);
      int it = 0;
      for (int i = qtiles.first(); ok && i < iend; i = qtiles.next(i + 1), ++it) {
        ok = mbar_wait(&qdo_full, it & 1, &abort_flag, p.status, 502);
        if (ok && it > 0) ok = mbar_wait(&dq_free, (it - 1) & 1, &abort_flag, p.status, 503);
        if (!ok) break;
        tc_fence_after();
        // S^T = K Q^T and dP^T = V dO^T  (K-major operands, K dimension = d)
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t koff = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
          mma_ss(tmem + C::kColS, sdesc_sw128(sK + koff, 16, 1024), sdesc_sw128(sQ + koff, 16, 1024),
                 idesc_s, ks > 0);
          mma_ss(tmem + C::kColDP, sdesc_sw128(sV + koff, 16, 1024),
                 sdesc_sw128(sDO + koff, 16, 1024), idesc_s, ks > 0);
        }
        mma_commit(&s_full);
        ok = mbar_wait(&p_full, it & 1, &abort_flag, p.status, 504);
        if (!ok) break;
        tc_fence_after();
        // dV += P^T dO, dK += dS^T Q   (A K-major over queries, B MN-major)
        // dQ  = dS K                   (A = dS^T read MN-major, B = K MN-major)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t aoff = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
          const uint32_t moff = ks * 2048;
          const uint32_t acc = (it > 0 || ks > 0) ? 1u : 0u;
          mma_ss(tmem + C::kColDV, sdesc_sw128(sP + aoff, 16, 1024),
                 sdesc_sw128(sDO + moff, C::kChunkBytes, 1024), idesc_acc, acc);
          mma_ss(tmem + C::kColDK, sdesc_sw128(sDS + aoff, 16, 1024),
                 sdesc_sw128(sQ + moff, C::kChunkBytes, 1024), idesc_acc, acc);
          mma_ss(tmem + C::kColDQ, sdesc_sw128(sDS + moff, C::kChunkBytes, 1024),
                 sdesc_sw128(sK + moff, C::kChunkBytes, 1024), idesc_dq, ks > 0);
        }
        mma_commit(&mma_done);
        mma_commit(&qdo_empty);
      }
      mma_commit(&drain);
      mbar_drain(&drain, 0);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int key = kt * 128 + tid;  // key row of this thread
    const bool key_live = key < kv_limit;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t sP = smem_addr(smem + C::kOffP), sDS = smem_addr(smem + C::kOffDS);
    const size_t head_row0 = (size_t)bh * p.N;
    int it = 0;
    bool ok = true;
    for (int i = qtiles.first(); i < iend; i = qtiles.next(i + 1), ++it) {
      const int buf = it & 1;
      {
        const int q = i * 128 + tid;
        float l2 = INFINITY, dd = 0.f;
        if (q < p.N) {
          const float l = p.lse[head_row0 + q];
          if (l != -INFINITY) l2 = l * kLog2e;  // empty rows keep +inf: P = 0
          dd = p.Dvec[head_row0 + q];
        }
        s_lse2[buf][tid] = l2;
        s_D[buf][tid] = dd;
      }
      mbar_arrive(&stats_ready[buf]);
      ok = mbar_wait_warp(&stats_ready[buf], (it >> 1) & 1, &abort_flag, p.status, 600);
      if (!ok) break;
      ok = mbar_wait_warp(&s_full, it & 1, &abort_flag, p.status, 601);
      if (!ok) break;
      tc_fence_after();
      const int q0 = i * 128;
      const bool need_causal = p.causal && (q0 < kt * 128 + 127);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {  // 32 query columns at a time
        uint32_t rs[32], rp[32];
        FA_TMEM_LD32_SYNC(tmem + C::kColS + lane_off + c * 32, rs);
        FA_TMEM_LD32_SYNC(tmem + C::kColDP + lane_off + c * 32, rp);
        uint32_t pp[16], dp[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float pv[2], dv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int qc = c * 32 + e + u;
            float pr = ex2(fmaf(__uint_as_float(rs[e + u]), p.scale_log2, -s_lse2[buf][qc]));
            if (!key_live || (need_causal && key > q0 + qc)) pr = 0.f;
            pv[u] = pr;
            dv[u] = p.scale * pr * (__uint_as_float(rp[e + u]) - s_D[buf][qc]);
          }
          pp[e / 2] = pack_bf16(pv[0], pv[1]);
          dp[e / 2] = pack_bf16(dv[0], dv[1]);
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int col = c * 32 + g * 8;
          const uint32_t off = (col >> 6) * C::kChunkBytes + sw128_offset(tid, col & 63);
          st_shared_v4(sP + off, pp[4 * g], pp[4 * g + 1], pp[4 * g + 2], pp[4 * g + 3]);
          st_shared_v4(sDS + off, dp[4 * g], dp[4 * g + 1], dp[4 * g + 2], dp[4 * g + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full);
      ok = mbar_wait_warp(&mma_done, it & 1, &abort_flag, p.status, 602);
      if (!ok) break;
      tc_fence_after();
      // dQ_i rows (lanes are query rows here) into the fp32 accumulator
      const int q = q0 + tid;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        FA_TMEM_LD32_SYNC(tmem + C::kColDQ + lane_off + c * 32, r);
        if (q < p.N) {
          float* dst = p.dq_acc + (head_row0 + q) * D + c * 32;
#pragma unroll
          for (int g = 0; g < 8; ++g)
            red_add_v4(dst + 4 * g, __uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                       __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
        }
      }
      tc_fence_before();
      mbar_arrive(&dq_free);
    }
    // ------------------------------------------------------------ dK, dV out
    // the TMEM loads are warp-collective: every lane takes part, only the
    // stores are limited to rows inside the sequence
    const bool live = __all_sync(0xffffffffu, ok && !abort_flag);
    if (live) {
      const size_t base = (head_row0 + key) * D;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* out = which == 0 ? p.dv : p.dk;
        const uint32_t col0 = which == 0 ? C::kColDV : C::kColDK;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          if (it > 0) {
            FA_TMEM_LD32_SYNC(tmem + col0 + lane_off + c * 32, r);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = 0u;
          }
          if (key < p.N) {
            uint4* dst = reinterpret_cast<uint4*>(out + base + c * 32);
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
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_dkdv_d(const BwdArgs& a, cudaStream_t s) {
  using C = BwdCfg<D>;
  const int BH = a.B * a.H;
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_bhnd_map(&mq, a.q, BH, a.N, D, 128) || !encode_bhnd_map(&mk, a.k, BH, a.N, D, 128) ||
      !encode_bhnd_map(&mv, a.v, BH, a.N, D, 128) || !encode_bhnd_map(&mdo, a.dO, BH, a.N, D, 128))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.lse = a.lse;
  p.Dvec = a.D;
  p.dq_acc = a.dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.kv_len = a.mask_kind == FA_MASK_KEY_PADDING ? a.kv_len : nullptr;
  p.block_mask = a.mask_kind == FA_MASK_BLOCK_SPARSE ? a.block_mask : nullptr;
  p.H = a.H;
  p.N = a.N;
  p.T = tiles_of(a.N, 128);
  p.BH = BH;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.causal = a.causal;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(fa_bwd_dkdv_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  fa_bwd_dkdv_kernel<D><<<p.T * BH, 192, C::kSmem, s>>>(mq, mk, mv, mdo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_bf16(const BwdArgs& a, cudaStream_t s) {
  return a.d == 64 ? launch_dkdv_d<64>(a, s) : launch_dkdv_d<128>(a, s);
}

}  // namespace fa
