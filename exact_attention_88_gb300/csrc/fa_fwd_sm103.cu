// Forward pass of exact attention on sm_103a tensor cores.
//
// One CTA computes a 128-row query tile Q_i of one (batch, head) against the
// visible 128-key tiles K_j, V_j with the online-softmax recurrence
// ("FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness", summary page, "Method": block statistics m~, P~, l~ merged
// into running m, l and the rescaled output O; blog review "From Online
// Softmax to FlashAttention", "Algorithm FlashAttention (Tiling)").  The
// division by l is deferred to the end, which is the same quantity.
//
// Roles (192 threads, two CTAs per SM so that one CTA's softmax overlaps the
// other's MMAs):
//   warps 0-3  softmax: thread t owns query row t of the tile (TMEM lane t);
//              reads S_ij from TMEM twice (row max, then exponentials), masks,
//              updates m and l, writes P~ = 2^(c S - m) as packed bf16 over the
//              S columns it has read, rescales O in TMEM when m grew by more
//              than 8 in log2 units (lazy rescale), and finally writes O / l and
//              lse.
//   warp 4     TMA producer: Q_i once, then K_j / V_j into rings of stages.
//   warp 5     MMA issuer (one thread): S = Q K^T into TMEM columns [0,128),
//              O += P V into TMEM columns [128, 128+d) with P read from TMEM.
// Scores are kept in base 2: c = scale * log2(e); lse = ln2 * (m + log2 l).
#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P~ stays below 2^8

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / 64;             // 64-column (128-byte) chunks
  static constexpr int kTileBytes = 128 * D * 2;     // one Q, K or V tile
  static constexpr int kChunkBytes = 128 * 128;      // 128 rows x 128 bytes
  static constexpr int kStages = (D == 64) ? 2 : 1;  // K/V ring depth (two CTAs per SM)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kSmem = kOffV + kStages * kTileBytes + 1024;  // + alignment slack
  static constexpr int kTmemCols = 256;              // S / P: [0,128), O: [128, 128+D)
  static constexpr int kThreads = 192;
};

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  const int32_t* kv_len;
  const uint8_t* block_mask;
  int H, N, T, BH;
  float scale_log2;
  int causal;
  int* status;
};

// Visible key tiles of query tile qt: 0 <= j < jend, skipping tiles the
// block-sparse mask row drops.
struct TileIter {
  const uint8_t* row;  // block-mask row or nullptr
  int jend;
  __device__ int first() const { return next(0); }
  __device__ int next(int j) const {
    if (row)
      while (j < jend && row[j] == 0) ++j;
    return j;
  }
};

template <int D>
__global__ void __launch_bounds__(192, 2)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t q_full, s_full, p_full, o_done, drain;
  __shared__ uint64_t k_full[C::kStages], v_full[C::kStages], k_empty[C::kStages],
      v_empty[C::kStages];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heaviest query tiles first (causal rows near the end see the most keys)
  const int lin = blockIdx.x;
  const int qt = p.T - 1 - lin / p.BH;
  const int bh = lin % p.BH;
  const int b = bh / p.H;

  int kv_limit = p.N;
  if (p.kv_len) kv_limit = max(0, min(p.kv_len[b], p.N));
  int jend = (kv_limit + 127) / 128;
  if (p.causal) jend = min(jend, qt + 1);
  const TileIter tiles{p.block_mask ? p.block_mask + (size_t)qt * p.T : nullptr, jend};

  if (tid == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&s_full, 1);
    mbar_init(&p_full, 128);
    mbar_init(&o_done, 1);
    mbar_init(&drain, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(&tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      mbar_expect_tx(&q_full, C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_3d(&tmQ, &q_full, smem + C::kOffQ + c * C::kChunkBytes, c * 64, qt * 128, bh);
      int kcount[C::kStages] = {}, vcount[C::kStages] = {};
      int it = 0;
      bool ok = true;
      for (int j = tiles.first(); j < tiles.jend && ok; j = tiles.next(j + 1), ++it) {
        const int st = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        ok = mbar_wait(&k_empty[st], ph ^ 1, &abort_flag, p.status, 101);
        if (!ok) break;
        mbar_expect_tx(&k_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(&tmK, &k_full[st], smem + C::kOffK + st * C::kTileBytes + c * C::kChunkBytes,
                      c * 64, j * 128, bh);
        ++kcount[st];
        ok = mbar_wait(&v_empty[st], ph ^ 1, &abort_flag, p.status, 102);
        if (!ok) break;
        mbar_expect_tx(&v_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(&tmV, &v_full[st], smem + C::kOffV + st * C::kTileBytes + c * C::kChunkBytes,
                      c * 64, j * 128, bh);
        ++vcount[st];
      }
      // every issued copy must have landed before the CTA may exit
      mbar_drain(&q_full, 0);
      for (int s = 0; s < C::kStages; ++s) {
        if (kcount[s]) mbar_drain(&k_full[s], (kcount[s] - 1) & 1);
        if (vcount[s]) mbar_drain(&v_full[s], (vcount[s] - 1) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
      const uint32_t sQ = smem_addr(smem + C::kOffQ);
      const uint32_t sK = smem_addr(smem + C::kOffK);
      const uint32_t sV = smem_addr(smem + C::kOffV);
      bool ok = mbar_wait(&q_full, 0, &abort_flag, p.status, 201);
      int it = 0;
      for (int j = tiles.first(); ok && j < tiles.jend; j = tiles.next(j + 1), ++it) {
        const int st = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        ok = mbar_wait(&k_full[st], ph, &abort_flag, p.status, 202);
        // P of the previous tile sits in the S columns until its P V is done
        if (ok && it > 0) ok = mbar_wait(&o_done, (it - 1) & 1, &abort_flag, p.status, 203);
        if (!ok) break;
        tc_fence_after();
        const uint32_t kbase = sK + st * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t ad = sdesc_sw128(sQ + (ks >> 2) * C::kChunkBytes + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(kbase + (ks >> 2) * C::kChunkBytes + (ks & 3) * 32, 16, 1024);
          mma_ss(tS, ad, bd, idesc_qk, ks > 0 ? 1u : 0u);
        }
        mma_commit(&s_full);
        mma_commit(&k_empty[st]);
        ok = mbar_wait(&p_full, it & 1, &abort_flag, p.status, 204);
        if (ok) ok = mbar_wait(&v_full[st], ph, &abort_flag, p.status, 205);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vbase = sV + st * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // 128 keys, 16 per MMA; P packed 8 columns per step
          const uint64_t bd = sdesc_sw128(vbase + ks * 2048, C::kChunkBytes, 1024);
          mma_ts(tO, tS + ks * 8, bd, idesc_pv, (it > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(&o_done);
        mma_commit(&v_empty[st]);
      }
      // all MMAs issued by this thread are complete once `drain` flips
      mma_commit(&drain);
      mbar_drain(&drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int row = qt * 128 + tid;  // query index of this thread
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float m = -INFINITY, l = 0.f;
    int it = 0;
    bool ok = true;
    for (int j = tiles.first(); j < tiles.jend; j = tiles.next(j + 1), ++it) {
      ok = mbar_wait_warp(&s_full, it & 1, &abort_flag, p.status, 301);
      if (!ok) break;
      tc_fence_after();
      const int key0 = j * 128;
      const bool need_mask = (p.causal && (key0 + 127 > qt * 128)) || key0 + 128 > kv_limit;
      // pass 1: row maximum of the tile
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        FA_TMEM_LD32_SYNC(tS + lane_off + c * 32, r);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int key = key0 + c * 32 + e;
          const bool dead = need_mask && (key >= kv_limit || (p.causal && key > row));
          tmax = fmaxf(tmax, dead ? -INFINITY : __uint_as_float(r[e]));
        }
      }
      const float m_tile = tmax * p.scale_log2;
      const float m_new = fmaxf(m, m_tile);
      const bool grow = m_new > m + kRescaleThreshold;  // true when m = -inf, m_new finite
      float alpha = 1.f;
      if (grow) {
        alpha = (m == -INFINITY) ? 0.f : ex2(m - m_new);
        m = m_new;
      }
      const float m_sub = (m == -INFINITY) ? 0.f : m;
      // pass 2: P~ = 2^(c S - m), row sum, packed bf16 over columns already read
      float rowsum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        FA_TMEM_LD32_SYNC(tS + lane_off + c * 32, r);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float pv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int key = key0 + c * 32 + e + u;
            const bool dead = need_mask && (key >= kv_limit || (p.causal && key > row));
            pv[u] = dead ? 0.f : ex2(fmaf(__uint_as_float(r[e + u]), p.scale_log2, -m_sub));
            rowsum += pv[u];
          }
          pk[e / 2] = pack_bf16(pv[0], pv[1]);
        }
        FA_TMEM_ST16(tS + lane_off + c * 16, pk);
      }
      l = l * alpha + rowsum;
      // O holds the sum up to the previous tile (its P V is complete: S of this
      // tile was issued after it); rescale when the running max moved
      if (it > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          FA_TMEM_LD32_SYNC(tO + lane_off + c * 32, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          FA_TMEM_ST32(tO + lane_off + c * 32, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full);
    }
    // ------------------------------------------------------------ epilogue
    if (ok) {
      bool have = it > 0;
      if (have) {
        have = mbar_wait_warp(&o_done, (it - 1) & 1, &abort_flag, p.status, 304);
        tc_fence_after();
      }
      if (__all_sync(0xffffffffu, !abort_flag)) {  // warp-uniform: TMEM loads below
        const bool empty_row = !(l > 0.f);
        const float inv = empty_row ? 0.f : 1.f / l;
        const size_t base = ((size_t)bh * p.N + row) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          if (have) {
            FA_TMEM_LD32_SYNC(tO + lane_off + c * 32, r);
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
  if (warp == 5) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t s) {
  using C = FwdCfg<D>;
  const int BH = a.B * a.H;
  CUtensorMap mq, mk, mv;
  if (!encode_bhnd_map(&mq, a.q, BH, a.N, D, 128) || !encode_bhnd_map(&mk, a.k, BH, a.N, D, 128) ||
      !encode_bhnd_map(&mv, a.v, BH, a.N, D, 128))
    return cudaErrorInvalidValue;
  FwdParams p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.kv_len = a.mask_kind == FA_MASK_KEY_PADDING ? a.kv_len : nullptr;
  p.block_mask = a.mask_kind == FA_MASK_BLOCK_SPARSE ? a.block_mask : nullptr;
  p.H = a.H;
  p.N = a.N;
  p.T = tiles_of(a.N, 128);
  p.BH = BH;
  p.scale_log2 = a.scale * kLog2e;
  p.causal = a.causal;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.T * BH);
  fa_fwd_kernel<D><<<grid, C::kThreads, C::kSmem, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t s) {
  return a.d == 64 ? launch_fwd_d<64>(a, s) : launch_fwd_d<128>(a, s);
}

}  // namespace fa
