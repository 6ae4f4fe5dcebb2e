// The exported C ABI of libfa: argument validation (on the host, before any
// CUDA runtime call), TMA descriptor encoding, the device status block, and
// dispatch to the kernel launchers of the other translation units.
#include <math.h>

#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

// 4-int status block per device (a __device__ variable: no allocation).
__device__ int g_status[4];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

constexpr int kMaxDevices = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool scale_ok(float s) { return s > 0.f && s != INFINITY; }  // false for NaN too

fa_status check_sizes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if ((long long)B * H > 65535) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H * N * d > (1ll << 40)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Tiles of one block-mask row the kernels can hold as a shared-memory bitmap.
constexpr int kMaxMaskTiles = 4096;
static_assert(kMaxMaskTiles == kMaxTileOrder, "one limit on the block-mask side");

fa_status check_mask(const fa_mask* m, int N, int* kind, const int32_t** kv,
                     const uint8_t** bm, const int32_t** order) {
  *kind = FA_MASK_NONE;
  *kv = nullptr;
  *bm = nullptr;
  *order = nullptr;
  if (!m) return FA_OK;
  switch (m->kind) {
    case FA_MASK_NONE:
      return FA_OK;
    case FA_MASK_KEY_PADDING:
      if (!m->kv_len || !aligned4(m->kv_len)) return FA_ERR_INVALID_ARG;
      *kind = FA_MASK_KEY_PADDING;
      *kv = m->kv_len;
      return FA_OK;
    case FA_MASK_BLOCK_SPARSE:
      if (!m->block_mask) return FA_ERR_INVALID_ARG;
      if (m->block_size != 128) return FA_ERR_UNSUPPORTED;
      if (tiles_of(N, 128) > kMaxMaskTiles) return FA_ERR_UNSUPPORTED;
      if (m->tile_order && !aligned4(m->tile_order)) return FA_ERR_ALIGNMENT;
      *kind = FA_MASK_BLOCK_SPARSE;
      *bm = m->block_mask;
      *order = m->tile_order;
      return FA_OK;
    default:
      return FA_ERR_INVALID_ARG;
  }
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Validates the caller's layout of one [B,H,N,d] tensor of `esize`-byte
// elements (NULL: dense) and returns it with the stride of every size-1
// dimension replaced by d, a value the TMA descriptor accepts and no index
// ever multiplies by anything but 0.
fa_status check_layout(const fa_layout* in, int B, int H, int N, int d, int esize, Layout* out) {
  const Layout dl = dense_layout(H, N, d);
  const long long given[3] = {in ? (long long)in->batch : dl.b, in ? (long long)in->head : dl.h,
                              in ? (long long)in->row : dl.n};
  const int extent[3] = {B, H, N};
  long long r[3];
  for (int i = 0; i < 3; ++i) {
    if (extent[i] == 1) {
      r[i] = d;
      continue;
    }
    if (given[i] <= 0 || given[i] >= (1ll << 40) / esize) return FA_ERR_UNSUPPORTED;
    if ((given[i] * esize) % 16 != 0) return FA_ERR_ALIGNMENT;
    r[i] = given[i];
  }
  if (N > 1 && r[2] < d) return FA_ERR_UNSUPPORTED;
  *out = Layout{r[0], r[1], r[2]};
  return FA_OK;
}

// Validates an additive bias: pointer 16-byte aligned, strides >= 0 and
// multiples of 4 elements (16 bytes: rows are read 4 floats at a time), the
// row stride 0 or >= N.
fa_status check_bias(const fa_bias* bias, int N, int esize, const float** ptr, Layout* lb) {
  *ptr = nullptr;
  *lb = Layout{0, 0, 0};
  if (!bias) return FA_OK;
  if (esize != 2) return FA_ERR_UNSUPPORTED;
  if (!bias->ptr) return FA_ERR_INVALID_ARG;
  if (!aligned16(bias->ptr)) return FA_ERR_ALIGNMENT;
  const long long st[3] = {(long long)bias->batch, (long long)bias->head, (long long)bias->row};
  for (long long x : st) {
    if (x < 0 || x >= (1ll << 40)) return FA_ERR_UNSUPPORTED;
    if (x % 4 != 0) return FA_ERR_ALIGNMENT;
  }
  if (st[2] != 0 && st[2] < N) return FA_ERR_UNSUPPORTED;
  *ptr = bias->ptr;
  *lb = Layout{st[0], st[1], st[2]};
  return FA_OK;
}

}  // namespace

// Validates a dropout request and derives the kernels' parameters: the
// 16-bit threshold t = min(65535, floor(p 65536 + 1/2)) (keep probability
// 1 - t/65536 exactly) and the scale 65536 / (65536 - t).  No request, or
// t = 0, is no dropout.
fa_status check_dropout(const fa_dropout* dr, int esize, DropParams* out) {
  *out = DropParams{0u, 0u, 0u, 0u, 1.f};
  if (!dr) return FA_OK;
  const float p = dr->p;
  if (!(p >= 0.f && p < 1.f)) return FA_ERR_INVALID_ARG;  // NaN fails too
  const double tt = floor((double)p * 65536.0 + 0.5);
  const uint32_t t = tt > 65535.0 ? 65535u : (uint32_t)tt;
  if (t == 0) return FA_OK;
  if (esize != 2) return FA_ERR_UNSUPPORTED;
  out->t = t;
  out->k0 = (uint32_t)(dr->seed & 0xFFFFFFFFull);
  out->k1 = (uint32_t)(dr->seed >> 32);
  out->offset = dr->offset;
  out->rp = (float)(65536.0 / (65536.0 - (double)t));
  return FA_OK;
}

bool encode_bhnd_map(CUtensorMap* map, const void* base, const Layout& l, int B, int H, int N,
                     int d, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)l.n * 2, (cuuint64_t)l.h * 2, (cuuint64_t)l.b * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_bwd_maps(const BwdArgs& a, CUtensorMap m[4]) {
  return encode_bhnd_map(&m[0], a.q, a.lq, a.B, a.H, a.N, a.d, 128) &&
         encode_bhnd_map(&m[1], a.k, a.lk, a.B, a.H, a.N, a.d, 128) &&
         encode_bhnd_map(&m[2], a.v, a.lv, a.B, a.H, a.N, a.d, 128) &&
         encode_bhnd_map(&m[3], a.dO, a.ldo, a.B, a.H, a.N, a.d, 128);
}

int* device_status() {
  static int* ptrs[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

}  // namespace fa

using namespace fa;

// Looked up only once every argument has been validated, so that argument
// errors are reported without touching the CUDA runtime.
template <typename Args>
static bool attach_status(Args* a) {
  a->status = device_status();
  return a->status != nullptr;
}

static fa_status fill_fwd(FwdArgs* a, const void* q, const void* k, const void* v, void* o,
                          float* lse, int B, int H, int N, int d, float scale, int causal,
                          const fa_mask* mask, const fa_options* opt, int esize) {
  fa_status st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  const fa_layouts* L = opt ? opt->layouts : nullptr;
  if ((st = check_dropout(opt ? opt->dropout : nullptr, esize, &a->drop)) != FA_OK) return st;
  if ((st = check_bias(opt ? opt->bias : nullptr, N, esize, &a->bias, &a->lb)) != FA_OK) return st;
  if ((st = check_layout(L ? &L->q : nullptr, B, H, N, d, esize, &a->lq)) != FA_OK ||
      (st = check_layout(L ? &L->k : nullptr, B, H, N, d, esize, &a->lk)) != FA_OK ||
      (st = check_layout(L ? &L->v : nullptr, B, H, N, d, esize, &a->lv)) != FA_OK ||
      (st = check_layout(L ? &L->o : nullptr, B, H, N, d, esize, &a->lo)) != FA_OK)
    return st;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse))
    return FA_ERR_ALIGNMENT;
  st = check_mask(mask, N, &a->mask_kind, &a->kv_len, &a->block_mask, &a->tile_order);
  if (st != FA_OK) return st;
  a->q = q; a->k = k; a->v = v; a->o = o; a->lse = lse;
  a->B = B; a->H = H; a->N = N; a->d = d;
  a->scale = scale;
  a->causal = causal;
  return FA_OK;
}

static fa_status fill_bwd_common(BwdArgs* a, int B, int H, int N, int d, float scale, int causal,
                                 const fa_mask* mask, const fa_options* opt = nullptr,
                                 int esize = 2) {
  fa_status st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  const fa_layouts* L = opt ? opt->layouts : nullptr;
  if ((st = check_dropout(opt ? opt->dropout : nullptr, esize, &a->drop)) != FA_OK) return st;
  if ((st = check_bias(opt ? opt->bias : nullptr, N, esize, &a->bias, &a->lb)) != FA_OK) return st;
  const fa_layout* in[8] = {L ? &L->q : nullptr,  L ? &L->k : nullptr,  L ? &L->v : nullptr,
                            L ? &L->o : nullptr,  L ? &L->dO : nullptr, L ? &L->dq : nullptr,
                            L ? &L->dk : nullptr, L ? &L->dv : nullptr};
  Layout* out[8] = {&a->lq, &a->lk, &a->lv, &a->lo, &a->ldo, &a->ldq, &a->ldk, &a->ldv};
  for (int t = 0; t < 8; ++t)
    if ((st = check_layout(in[t], B, H, N, d, esize, out[t])) != FA_OK) return st;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  st = check_mask(mask, N, &a->mask_kind, &a->kv_len, &a->block_mask, &a->tile_order);
  if (st != FA_OK) return st;
  a->B = B; a->H = H; a->N = N; a->d = d;
  a->scale = scale;
  a->causal = causal;
  return FA_OK;
}

// The workspace: D (fp32 [B,H,N], padded to 256 bytes), then the work
// counter of the persistent backward kernel.
constexpr size_t kSchedBytes = 256;

static fa_status split_workspace(BwdArgs* a, void* ws, size_t ws_bytes) {
  if (!ws) return FA_ERR_WORKSPACE;
  if (!aligned16(ws)) return FA_ERR_ALIGNMENT;
  const size_t d_bytes = round256((size_t)a->B * a->H * a->N * sizeof(float));
  if (ws_bytes < d_bytes + kSchedBytes) return FA_ERR_WORKSPACE;
  a->D = static_cast<float*>(ws);
  a->sched = reinterpret_cast<int*>(static_cast<char*>(ws) + d_bytes);
  return FA_OK;
}

// Validation shared by the whole-backward calls (bf16: esize 2, fp32: 4).
static fa_status fill_bwd_full(BwdArgs* a, const void* q, const void* k, const void* v,
                               const void* o, const void* dO, const float* lse, void* dq,
                               void* dk, void* dv, void* workspace, size_t workspace_bytes, int B,
                               int H, int N, int d, float scale, int causal, const fa_mask* mask,
                               const fa_options* opt, int esize) {
  fa_status st = fill_bwd_common(a, B, H, N, d, scale, causal, mask, opt, esize);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned4(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_ALIGNMENT;
  st = split_workspace(a, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  a->q = q; a->k = k; a->v = v; a->o = o; a->dO = dO; a->lse = lse;
  a->dq = dq; a->dk = dk; a->dv = dv;
  return attach_status(a) ? FA_OK : FA_ERR_CUDA;
}

int fa::device_sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev] = sms;
  return sms;
}

// Text of the last CUDA error a call of this thread failed with.
static thread_local const char* t_last_cuda_error = "no CUDA error";

static fa_status launched(cudaError_t e) {
  if (e == cudaSuccess) return FA_OK;
  t_last_cuda_error = cudaGetErrorString(e);
  return FA_ERR_CUDA;
}

fa_status fa::cuda_status(cudaError_t e) { return launched(e); }

fa_status fa::check_bwd_args(const void* q, const void* k, const void* v, const void* o,
                             const void* dO, const float* lse, void* dq, void* dk, void* dv,
                             int B, int H, int N, int d, float scale, int causal,
                             const fa_mask* mask) {
  BwdArgs a{};
  fa_status st = fill_bwd_common(&a, B, H, N, d, scale, causal, mask);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned4(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_ALIGNMENT;
  return FA_OK;
}

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported size or option";
    case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT: tensor pointer not 16-byte aligned";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing or too small";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel wait gave up";
  }
  return "unknown fa_status";
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_sizes(B, H, N, d) != FA_OK) return 0;
  return round256((size_t)B * H * N * sizeof(float)) + kSchedBytes;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, const fa_mask* mask, void* stream) {
  return fa_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, mask, nullptr, stream);
}

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                    int N, int d, float scale, int causal, const fa_mask* mask,
                    const fa_options* options, void* stream) {
  FwdArgs a{};
  fa_status st = fill_fwd(&a, q, k, v, o, lse, B, H, N, d, scale, causal, mask, options, 2);
  if (st != FA_OK) return st;
  if (!attach_status(&a)) return FA_ERR_CUDA;
  return launched(launch_fwd_bf16(a, static_cast<cudaStream_t>(stream)));
}

fa_status fa_fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                      int H, int N, int d, float scale, int causal, const fa_mask* mask,
                      void* stream) {
  return fa_fwd_fp32_ex(q, k, v, o, lse, B, H, N, d, scale, causal, mask, nullptr, stream);
}

fa_status fa_fwd_fp32_ex(const float* q, const float* k, const float* v, float* o, float* lse,
                         int B, int H, int N, int d, float scale, int causal, const fa_mask* mask,
                         const fa_options* options, void* stream) {
  FwdArgs a{};
  fa_status st = fill_fwd(&a, q, k, v, o, lse, B, H, N, d, scale, causal, mask, options, 4);
  if (st != FA_OK) return st;
  if (!attach_status(&a)) return FA_ERR_CUDA;
  return launched(launch_fwd_fp32(a, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace,
                 size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                 const fa_mask* mask, void* stream) {
  return fa_bwd_ex(q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale,
                   causal, mask, nullptr, stream);
}

fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dO,
                    const float* lse, void* dq, void* dk, void* dv, void* workspace,
                    size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                    const fa_mask* mask, const fa_options* options, void* stream) {
  BwdArgs a{};
  fa_status st = fill_bwd_full(&a, q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B,
                               H, N, d, scale, causal, mask, options, 2);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = launched(launch_bwd_preprocess(a, s));
  // dK/dV and dQ in one launch, their CTAs interleaved
  if (st == FA_OK) st = launched(launch_bwd_pair_bf16(a, s));
  return st;
}

fa_status fa_bwd_preprocess(const void* o, const void* dO, float* D, int B, int H, int N, int d,
                            void* stream) {
  return fa_bwd_preprocess_ex(o, dO, D, B, H, N, d, nullptr, stream);
}

fa_status fa_bwd_preprocess_ex(const void* o, const void* dO, float* D, int B, int H, int N, int d,
                               const fa_options* options, void* stream) {
  BwdArgs a{};
  fa_status st = fill_bwd_common(&a, B, H, N, d, 1.0f, 0, nullptr, options);
  if (st != FA_OK) return st;
  if (!o || !dO || !D) return FA_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dO) || !aligned4(D)) return FA_ERR_ALIGNMENT;
  a.o = o; a.dO = dO; a.D = D;
  if (!attach_status(&a)) return FA_ERR_CUDA;
  return launched(launch_bwd_preprocess(a, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO,
                      const float* lse, const float* D, void* dk, void* dv, int B, int H, int N,
                      int d, float scale, int causal, const fa_mask* mask, void* stream) {
  return fa_bwd_dkdv_ex(q, k, v, dO, lse, D, dk, dv, B, H, N, d, scale, causal, mask, nullptr,
                        stream);
}

fa_status fa_bwd_dkdv_ex(const void* q, const void* k, const void* v, const void* dO,
                         const float* lse, const float* D, void* dk, void* dv, int B, int H,
                         int N, int d, float scale, int causal, const fa_mask* mask,
                         const fa_options* options, void* stream) {
  BwdArgs a{};
  fa_status st = fill_bwd_common(&a, B, H, N, d, scale, causal, mask, options);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !dO || !lse || !D || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned4(lse) ||
      !aligned4(D) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_ALIGNMENT;
  a.q = q; a.k = k; a.v = v; a.dO = dO; a.lse = lse;
  a.D = const_cast<float*>(D); a.dk = dk; a.dv = dv;
  if (!attach_status(&a)) return FA_ERR_CUDA;
  return launched(launch_bwd_dkdv_bf16(a, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                    const float* D, void* dq, int B, int H, int N, int d, float scale, int causal,
                    const fa_mask* mask, void* stream) {
  return fa_bwd_dq_ex(q, k, v, dO, lse, D, dq, B, H, N, d, scale, causal, mask, nullptr, stream);
}

fa_status fa_bwd_dq_ex(const void* q, const void* k, const void* v, const void* dO,
                       const float* lse, const float* D, void* dq, int B, int H, int N, int d,
                       float scale, int causal, const fa_mask* mask, const fa_options* options,
                       void* stream) {
  BwdArgs a{};
  fa_status st = fill_bwd_common(&a, B, H, N, d, scale, causal, mask, options);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !dO || !lse || !D || !dq) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned4(lse) ||
      !aligned4(D) || !aligned16(dq))
    return FA_ERR_ALIGNMENT;
  a.q = q; a.k = k; a.v = v; a.dO = dO; a.lse = lse;
  a.D = const_cast<float*>(D); a.dq = dq;
  if (!attach_status(&a)) return FA_ERR_CUDA;
  return launched(launch_bwd_dq_bf16(a, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd_fp32(const float* q, const float* k, const float* v, const float* o,
                      const float* dO, const float* lse, float* dq, float* dk, float* dv,
                      void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                      float scale, int causal, const fa_mask* mask, void* stream) {
  return fa_bwd_fp32_ex(q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d,
                        scale, causal, mask, nullptr, stream);
}

fa_status fa_bwd_fp32_ex(const float* q, const float* k, const float* v, const float* o,
                         const float* dO, const float* lse, float* dq, float* dk, float* dv,
                         void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                         float scale, int causal, const fa_mask* mask, const fa_options* options,
                         void* stream) {
  BwdArgs a{};
  fa_status st = fill_bwd_full(&a, q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B,
                               H, N, d, scale, causal, mask, options, 4);
  if (st != FA_OK) return st;
  return launched(launch_bwd_fp32(a, static_cast<cudaStream_t>(stream)));
}

int fa_block_mask_order_len(int T) { return tile_order_len(T); }

fa_status fa_block_mask_order(const uint8_t* block_mask, int T, int causal, int32_t* tile_order,
                              void* stream) {
  if (!block_mask || !tile_order || tile_order_len(T) == 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!aligned4(tile_order)) return FA_ERR_ALIGNMENT;
  return launched(
      launch_tile_order(block_mask, T, causal, tile_order, static_cast<cudaStream_t>(stream)));
}

const char* fa_last_cuda_error(void) { return t_last_cuda_error; }

fa_status fa_get_device_status(void* stream, int* site) {
  if (site) *site = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int* st = device_status();
  if (!st) return FA_ERR_CUDA;
  int h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, st, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (h[0] != 0) {
    if (site) *site = h[1];
    const int z[4] = {0, 0, 0, 0};
    if (cudaMemcpy(st, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    return h[0] == kStatusTimeoutCode ? FA_ERR_TIMEOUT : FA_ERR_CUDA;
  }
  return FA_OK;
}

fa_status fa_debug_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return FA_ERR_INVALID_ARG;
  int* st = device_status();
  if (!st) return FA_ERR_CUDA;
  return launched(launch_wait_probe(1000ull * limit_us, st, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
