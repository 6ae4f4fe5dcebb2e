/*
 * fa.h -- C ABI of libfa, exact attention for NVIDIA GB300 (sm_103a).
 *
 * Computes, for every batch element b and head h (the plain definition of
 * attention: "FlashAttention: Fast and Memory-Efficient Exact Attention with
 * IO-Awareness", summary page, "Problem and motivation"; scale on the scores
 * as in the GitHub issue "Fewer matrix multiplications, same results"):
 *
 *     S   = scale * Q K^T      (entries of invisible keys are -inf)
 *     P   = softmax(S)         (row-wise, with the row maximum subtracted)
 *     O   = P V
 *     lse = ln sum_j exp(S_ij)  (natural log; the only statistic kept)
 *
 * tile by tile with the online-softmax recurrence (blog review "From Online
 * Softmax to FlashAttention", "Algorithm FlashAttention (Tiling)"; summary
 * page, "Method": running max m, running denominator l, rescaled output), so
 * the N x N score matrix never reaches device memory, and the backward pass
 * recomputes P on chip from Q, K and lse (summary page, "Key ideas:
 * recomputation in the backward pass").
 *
 * Conventions shared by every call:
 *   - Tensors are dense row-major [B, H, N, d] (d contiguous) in DEVICE
 *     memory, 16-byte aligned; lse and D are fp32 [B, H, N].  The *_ex
 *     calls take Q, K, V, O, dO, dQ, dK, dV in any layout whose d elements of
 *     a row are contiguous (fa_layout), and dropout (fa_dropout); lse and D
 *     stay dense.  The caller owns
 *     every buffer; the library allocates nothing.
 *   - bf16 calls take bf16 (uint16 storage) Q, K, V, O, dO, dQ, dK, dV and
 *     accumulate in fp32.  *_fp32 calls take fp32 everywhere.
 *   - d must be 64 or 128; N >= 1 (any N: ragged tails are masked); B >= 1,
 *     H >= 1, B*H <= 65535; scale must be positive and finite.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous with respect to the host, like cuBLAS: a returned
 *     FA_OK means the work was enqueued.
 *   - Argument errors are detected on the host before anything is launched
 *     (and before any CUDA runtime call), and reported through the return
 *     value only.
 *   - Masking: `causal` keeps keys j <= i (queries and keys share indices).
 *     `mask` may add key padding (keys j >= kv_len[b] are invisible) or a
 *     block-sparse tile mask (tile (i/128, j/128) visible iff
 *     block_mask[(i/128)*T + j/128] != 0, T = ceil(N/128); summary page,
 *     "Extension: block-sparse FlashAttention").  causal combines with either
 *     (intersection).  A query row with no visible key gets O = 0,
 *     lse = -inf and contributes no gradient.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, bad mask kind  */
  FA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (d not 64/128, ...)   */
  FA_ERR_ALIGNMENT = 3,    /* a tensor pointer is not 16-byte aligned         */
  FA_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required      */
  FA_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed               */
  FA_ERR_TIMEOUT = 6       /* a kernel gave up waiting (see fa_get_device_status) */
} fa_status;

typedef enum {
  FA_MASK_NONE = 0,
  FA_MASK_KEY_PADDING = 1,
  FA_MASK_BLOCK_SPARSE = 2
} fa_mask_kind;

typedef struct {
  int kind;                  /* an fa_mask_kind                                     */
  const int32_t* kv_len;     /* KEY_PADDING: device int32 [B]; values are clamped   */
                             /* to 0..N (0 = every key of the batch is padding)     */
  const uint8_t* block_mask; /* BLOCK_SPARSE: device uint8 [T*T], T = ceil(N/128)   */
                             /* <= 4096 (N <= 524288; FA_ERR_UNSUPPORTED beyond)    */
  int block_size;            /* BLOCK_SPARSE: tile edge of block_mask, must be 128  */
  const int32_t* tile_order; /* BLOCK_SPARSE, optional (NULL: the default order):    */
                             /* the work order fa_block_mask_order wrote for this   */
                             /* block_mask; device int32, 4-byte aligned            */
} fa_mask;

/* Work order of a block-sparse mask.  The kernels skip the tiles the mask
 * hides (summary page, "Extension: block-sparse FlashAttention": only the
 * nonzero blocks are visited) and give each CTA one tile row or column, so a
 * row or column that sees far more tiles than the rest (a global token) ends
 * the kernel alone if the grid takes it last.  This call writes, on `stream`,
 * fa_block_mask_order_len(T) int32 to tile_order:
 *   [0, T)              query tiles, most visible key tiles first
 *   [T, 2T)             key tiles, most query tiles that see them first
 * counting with the causal restriction when causal = 1; ties keep the lower
 * index first.  Passed as fa_mask.tile_order, the kernels take their tiles in
 * that order; every tile is still computed exactly once and the results are
 * bit-identical to the default order's.  The buffer must be this call's
 * output (any other permutation of each part is also correct; contents that
 * are not permutations leave output tiles unwritten or written twice -- the
 * kernels only clamp entries to [0, T)).  Recompute it when the mask changes;
 * it costs one small launch per mask.
 *   block_mask : device uint8 [T*T].   T : 1..4096.   causal : 0 or 1.
 * Argument errors come back before any CUDA runtime call. */
int fa_block_mask_order_len(int T); /* 2T + (T+1)/2, or 0 when T is out of range */
fa_status fa_block_mask_order(const uint8_t* block_mask, int T, int causal, int32_t* tile_order,
                              void* stream);

/* Forward pass, bf16 in/out.
 *   q, k, v : [B,H,N,d] bf16 inputs.   o : [B,H,N,d] bf16 output.
 *   lse     : [B,H,N] fp32 output, natural-log log-sum-exp of each score row
 *             (-inf for a row with no visible key).
 *   scale   : multiplies Q K^T (1/sqrt(d) for standard attention).
 *   causal  : 0 or 1.   mask : NULL for none.
 * Summary page "Method" (block statistics m, l and the rescaled output) and
 * blog review "Algorithm FlashAttention (Tiling)". */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, const fa_mask* mask, void* stream);

/* Bytes of device workspace fa_bwd / fa_bwd_fp32 need: D (fp32 [B,H,N]),
 * padded to 256 bytes, then 256 bytes for the counter from which the backward
 * kernel's CTAs take their units of work.  0 on bad sizes. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/* Backward pass, bf16.  Given the forward's inputs, its outputs o and lse,
 * and the output gradient dO, writes dq, dk, dv ([B,H,N,d] bf16) for the loss
 * whose gradient with respect to O is dO.  P is recomputed from q, k, lse
 * (summary page, "Key ideas: recomputation in the backward pass"); the
 * gradient formulas (dV = P^T dO, dP = dO V^T, D = rowsum(dO o O),
 * dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q) are the textbook
 * derivative, which the pages do not write out.
 *   workspace : device, >= fa_bwd_workspace_size(B,H,N,d) bytes, 16-byte
 *               aligned; contents on entry are ignored.
 * Runs fa_bwd_preprocess, fa_bwd_dkdv and fa_bwd_dq on `stream`. */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace,
                 size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                 const fa_mask* mask, void* stream);

/* The three steps of fa_bwd, exposed for timing each kernel on its own.
 * fa_bwd_preprocess: D[b,h,i] = sum_c dO[b,h,i,c] * O[b,h,i,c] (fp32 [B,H,N]).
 * fa_bwd_dkdv: recomputes P and dS tile by tile for each 128-key tile and
 *   writes dk, dv (bf16 [B,H,N,d]).  D as left by the preprocess.
 * fa_bwd_dq: recomputes P and dS tile by tile for each 128-query tile and
 *   writes dq (bf16 [B,H,N,d]); each row of dq is summed by one CTA in fp32,
 *   so dq is the same bit for bit from run to run.
 * fa_bwd_dkdv and fa_bwd_dq read the same inputs and write disjoint outputs:
 *   they may run in either order, or concurrently on two streams. */
fa_status fa_bwd_preprocess(const void* o, const void* dO, float* D, int B, int H, int N, int d,
                            void* stream);
fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO,
                      const float* lse, const float* D, void* dk, void* dv, int B, int H, int N,
                      int d, float scale, int causal, const fa_mask* mask, void* stream);
fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                    const float* D, void* dq, int B, int H, int N, int d, float scale, int causal,
                    const fa_mask* mask, void* stream);

/* fp32 twins of fa_fwd / fa_bwd: identical argument meaning with fp32
 * tensors everywhere (CUDA cores, no tensor cores; for small fp32 workloads). */
fa_status fa_fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                      int H, int N, int d, float scale, int causal, const fa_mask* mask,
                      void* stream);
fa_status fa_bwd_fp32(const float* q, const float* k, const float* v, const float* o,
                      const float* dO, const float* lse, float* dq, float* dk, float* dv,
                      void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                      float scale, int causal, const fa_mask* mask, void* stream);

/* Layout of one [B, H, N, d] tensor as element strides: element (b, h, n, c)
 * is at base + b*batch + h*head + n*row + c (the d elements of a row are
 * contiguous).  Dense [B,H,N,d] is {H*N*d, N*d, d}; a [B,N,H,d] buffer (the
 * heads of a packed projection side by side in each row) read as [B,H,N,d]
 * is {N*H*d, d, H*d}.  Rules, checked on the host before any launch:
 *   - the stride of a dimension of size 1 is ignored;
 *   - every other stride is positive (FA_ERR_UNSUPPORTED otherwise), a
 *     multiple of 16 bytes (8 bf16 or 4 fp32 elements; FA_ERR_ALIGNMENT
 *     otherwise) and below 2^40 bytes (FA_ERR_UNSUPPORTED otherwise);
 *   - the row stride is at least d when N > 1 (FA_ERR_UNSUPPORTED).
 * An output must not overlap another tensor of the same call; this is not
 * checked. */
typedef struct {
  int64_t batch, head, row;
} fa_layout;

/* Layouts of the tensors of one call.  The forward reads q, k, v, o and
 * ignores the rest. */
typedef struct {
  fa_layout q, k, v, o, dO, dq, dk, dv;
} fa_layouts;

/* Dropout on the attention probabilities.  The summary page lists dropout
 * among the operations fused into the attention kernel and says that the
 * backward pass keeps the generator's state to regenerate the mask on chip
 * ("Key ideas: kernel fusion"; its question on the auxiliary memory of the
 * backward pass).  Reading: with Z_ij in {0, 1} kept with probability 1 - p,
 *     O = (P o Z) V / (1 - p),   lse of the undropped scores,
 * and the backward is the chain rule through it (dV = (P o Z)^T dO / (1-p),
 * dS = P o (Z o dO V^T / (1-p) - D), D = rowsum(dO o O) as without dropout).
 * Z is drawn from Philox4x32-10 (Salmon et al., "Parallel random numbers: as
 * easy as 1, 2, 3", SC 2011): element (i, j) of head (b, h) takes the call
 * with counter (j / 8, i, b*H + h, offset) and key (seed & 0xFFFFFFFF,
 * seed >> 32); of its four output words, key j takes the low (j even) or
 * high (j odd) 16 bits of word (j % 8) / 2 and is kept when they are >= t,
 * t = min(65535, floor(p * 65536 + 0.5)) -- so the keep probability is
 * exactly 1 - t/65536 and the kept entries are scaled by 65536 / (65536 - t).
 * The forward and backward of one step must use the same p, seed, offset. */
typedef struct {
  float p;          /* drop probability, 0 <= p < 1 (0: no dropout)          */
  uint64_t seed;    /* generator key                                         */
  uint32_t offset;  /* fourth counter word: a new value per step (e.g. the step number) */
} fa_dropout;

/* Additive score bias: the "+ mask" term of the scores as a tensor,
 *     S_ij = scale q_i . k_j + bias[b, h, i, j]
 * added before the causal / padding / block masks (summary page, "Problem
 * and motivation"; the masks of the glossary page "Flash Attention",
 * "Normalization and Masking").  fp32 in device memory; element (b, h, i, j)
 * at ptr + b*batch + h*head + i*row + j.  A stride of 0 broadcasts (one
 * [N, N] bias for every head: batch = head = 0).  -inf hides a key; +inf
 * and NaN are not allowed.  Rules: ptr 16-byte aligned; strides >= 0,
 * multiples of 4 elements, row >= N unless 0 (FA_ERR_ALIGNMENT /
 * FA_ERR_UNSUPPORTED otherwise).  The bias receives no gradient. */
typedef struct {
  const float* ptr;
  int64_t batch, head, row;
} fa_bias;

/* Options of the *_ex calls.  NULL options, or NULL members, mean dense
 * tensors, no dropout and no bias. */
typedef struct {
  const fa_layouts* layouts;
  const fa_dropout* dropout;  /* bf16 calls only: FA_ERR_UNSUPPORTED for fp32 */
  const fa_bias* bias;        /* bf16 calls only: FA_ERR_UNSUPPORTED for fp32 */
} fa_options;

/* fa_fwd / fa_bwd / fa_fwd_fp32 / fa_bwd_fp32 and the three backward steps
 * with options; every other argument as in the plain call.  With dense
 * layouts and no dropout the work and results are those of the plain call;
 * other layouts give the same results on the same values (the kernels read
 * and write through the strides -- the TMA descriptors of the bf16 kernels
 * carry them -- and nothing is copied).  Errors: a p outside [0, 1)
 * (or NaN) is FA_ERR_INVALID_ARG; dropout or a bias on an fp32 call,
 * FA_ERR_UNSUPPORTED. */
fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                    int N, int d, float scale, int causal, const fa_mask* mask,
                    const fa_options* options, void* stream);
fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dO,
                    const float* lse, void* dq, void* dk, void* dv, void* workspace,
                    size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                    const fa_mask* mask, const fa_options* options, void* stream);
fa_status fa_fwd_fp32_ex(const float* q, const float* k, const float* v, float* o, float* lse,
                         int B, int H, int N, int d, float scale, int causal, const fa_mask* mask,
                         const fa_options* options, void* stream);
fa_status fa_bwd_fp32_ex(const float* q, const float* k, const float* v, const float* o,
                         const float* dO, const float* lse, float* dq, float* dk, float* dv,
                         void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                         float scale, int causal, const fa_mask* mask, const fa_options* options,
                         void* stream);
/* The backward steps with options (layouts of o, dO for the preprocess;
 * dropout and bias for fa_bwd_dkdv_ex and fa_bwd_dq_ex). */
fa_status fa_bwd_preprocess_ex(const void* o, const void* dO, float* D, int B, int H, int N, int d,
                               const fa_options* options, void* stream);
fa_status fa_bwd_dkdv_ex(const void* q, const void* k, const void* v, const void* dO,
                         const float* lse, const float* D, void* dk, void* dv, int B, int H,
                         int N, int d, float scale, int causal, const fa_mask* mask,
                         const fa_options* options, void* stream);
fa_status fa_bwd_dq_ex(const void* q, const void* k, const void* v, const void* dO,
                       const float* lse, const float* D, void* dq, int B, int H, int N, int d,
                       float scale, int causal, const fa_mask* mask, const fa_options* options,
                       void* stream);

/* Size of the fixed scratch array fa_bwd_noalloc works in: 32 MiB. */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)

/* fa_bwd for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call.  fa_bwd needs a caller-allocated workspace; some
 * callers cannot provide one, for example a plugin inside a host framework
 * that has reserved all device memory for its own pool and does not let
 * extensions call cudaMalloc, or latency-critical code that must avoid
 * cudaMalloc/cudaFree because they can synchronize the whole device.  This
 * call takes the workspace from a fixed array of FA_NOALLOC_SCRATCH_BYTES
 * compiled into the library (every GPU that loads the library holds it until
 * the process exits) and calls no allocator at all.
 *   Arguments and results are those of fa_bwd without the workspace pair;
 *   argument errors come back with fa_bwd's codes, from host-only checks
 *   made before any CUDA runtime call.
 *   Sizes whose workspace (fa_bwd_workspace_size) exceeds
 *   FA_NOALLOC_SCRATCH_BYTES are rejected with FA_ERR_UNSUPPORTED.
 *   The first call on a device looks up the array's device address (a CUDA
 *   runtime query, done once per device with that device current); make that
 *   first call before any stream capture.
 *   Every call shares the one array, which keeps the previous call's
 *   contents; each call rewrites what it needs before reading it.  Calls that
 *   overlap on the GPU (other streams, other host threads) race on the array:
 *   serialize them. */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale, int causal, const fa_mask* mask,
                         void* stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* fa_status_string(fa_status s);

/* Text of the CUDA error behind the last FA_ERR_CUDA that a launching call
 * of the calling thread returned ("no CUDA error" if none).  Static string. */
const char* fa_last_cuda_error(void);

/* Synchronizes `stream`, then reports and clears the device-side status that
 * the kernels raise when a wait inside them gives up (FA_ERR_TIMEOUT), or
 * FA_ERR_CUDA if the stream reports an error.  FA_OK otherwise.  If site is
 * not NULL it receives the id of the wait that gave up. */
fa_status fa_get_device_status(void* stream, int* site);

/* Diagnostic: launches one CTA that waits on an mbarrier no one arrives on,
 * with the given limit (1..1000000 microseconds), exactly as the attention
 * kernels bound their waits.  The kernel returns normally; a following
 * fa_get_device_status reports FA_ERR_TIMEOUT.  Lets the failure path be
 * checked without hanging or faulting a GPU. */
fa_status fa_debug_wait_timeout(unsigned int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
