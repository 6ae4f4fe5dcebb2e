"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: it draws random tensors, rounds
them to the storage precision, and draws masks and sample indices.  Both the
oracle-side tests and the GPU-side tests/bench take their inputs from here.

The workloads stand in for the workloads of the FlashAttention paper (summary
page "FlashAttention: Fast and Memory-Efficient Exact Attention with
IO-Awareness", section "Results": GPT-2 at sequence length 1K, BERT-large at
512, long-context causal models up to 64K tokens, block-sparse attention on
long sequences up to the 64K tokens of Path-256),
whose datasets and weights are not available: only the shapes, masks and value
distributions are reproduced.

Recipe (every workload, seed 0 unless stated):
  rng = numpy.random.default_rng(seed)  (PCG64)
  Q, K, V, dO = rng.standard_normal([B,H,N,d], float32) in that order,
  times `value_scale` (0.5 for the long causal workload: exact in binary),
  then rounded to bf16 with round-to-nearest-even (fp32 workloads keep fp32);
  then kv_len = rng.integers(128, 513, B)           (key-padding workload)
  then tile mask = rng.random((T, T)) < 0.125, diagonal forced to 1
                                    (block-sparse workloads, pattern "random";
                                     the other patterns draw nothing, see
                                     block_mask_pattern)
  then sampled rows: per (b, h), rng.choice(N, 256, replace=False) for query
  rows, then the same for key rows (long workloads only).
"""
import dataclasses
import hashlib
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "bf16" or "fp32"
    causal: bool
    mask: str             # "none", "key_padding", "block_sparse"
    value_scale: float = 1.0
    sampled: bool = False  # check on sampled rows instead of every row
    block: int = 128
    sparse_p: float = 0.125
    pattern: str = "random"  # tile-mask pattern of block-sparse workloads

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d)

    @property
    def tiles(self):
        return (self.N + self.block - 1) // self.block


WORKLOADS = {
    # tiny fp32 forward, run non-causal and causal
    "tiny_fp32": Workload("tiny_fp32", 1, 2, 256, 64, "fp32", False, "none"),
    "tiny_fp32_causal": Workload("tiny_fp32_causal", 1, 2, 256, 64, "fp32", True, "none"),
    # GPT-2-small-shaped causal self-attention
    "gpt2_causal": Workload("gpt2_causal", 8, 12, 1024, 64, "bf16", True, "none"),
    # BERT-large-shaped encoder attention with key padding
    "bert_padding": Workload("bert_padding", 16, 16, 512, 64, "bf16", False, "key_padding"),
    # long-context causal attention, head dim 128
    "long_causal_d128": Workload("long_causal_d128", 1, 16, 16384, 128, "bf16", True, "none",
                                 value_scale=0.5, sampled=True),
    # block-sparse attention on long sequences
    "block_sparse": Workload("block_sparse", 2, 16, 16384, 64, "bf16", False, "block_sparse",
                             sampled=True),
    # the same sequences under structured tile masks (the pages fix no pattern;
    # these are common fixed patterns, see block_mask_pattern)
    "sparse_local_global": Workload("sparse_local_global", 2, 16, 16384, 64, "bf16", False,
                                    "block_sparse", sampled=True, pattern="local_global"),
    "sparse_butterfly": Workload("sparse_butterfly", 2, 16, 16384, 64, "bf16", False,
                                 "block_sparse", sampled=True, pattern="butterfly"),
    # Path-256 length (a 256 x 256 image as 65536 tokens) under a butterfly mask
    "path256_butterfly": Workload("path256_butterfly", 1, 8, 65536, 64, "bf16", False,
                                  "block_sparse", sampled=True, pattern="butterfly"),
    # 64K-token causal context (the pages' longest dense sequences), head dim 128
    "causal_64k_d128": Workload("causal_64k_d128", 1, 4, 65536, 128, "bf16", True, "none",
                                value_scale=0.5, sampled=True),
}


def bf16_round(x):
    """Round float32 values to the nearest bf16 (ties to even); returns
    (float32 array holding the rounded values, uint16 bit patterns)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    back = (r.astype(np.uint32) << 16).view(np.float32)
    return back, r


def generate(w, seed=0, samples=256):
    """Draw the inputs of workload `w` (a Workload or its name).

    Returns a dict with float32 arrays q, k, v, do (values exactly
    representable in the storage dtype), for bf16 workloads the uint16 bit
    patterns q_bits..do_bits, kv_len (int32 [B] or None), block_mask (uint8
    [T,T] or None), and for sampled workloads int64 rows / cols [B,H,samples]."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    rng = np.random.default_rng(seed)
    shape = (w.B, w.H, w.N, w.d)
    out = {"workload": w}
    for name in ("q", "k", "v", "do"):
        x = rng.standard_normal(shape, dtype=np.float32)
        if w.value_scale != 1.0:
            x *= np.float32(w.value_scale)
        if w.dtype == "bf16":
            out[name], out[name + "_bits"] = bf16_round(x)
        else:
            out[name] = x
    out["kv_len"] = None
    out["block_mask"] = None
    if w.mask == "key_padding":
        out["kv_len"] = rng.integers(128, 513, w.B).astype(np.int32)
    if w.mask == "block_sparse":
        out["block_mask"] = block_mask_pattern(w.pattern, w.tiles, rng, w.sparse_p)
    if w.sampled:
        rows = np.zeros((w.B, w.H, samples), np.int64)
        cols = np.zeros((w.B, w.H, samples), np.int64)
        for b in range(w.B):
            for h in range(w.H):
                rows[b, h] = rng.choice(w.N, samples, replace=False)
        for b in range(w.B):
            for h in range(w.H):
                cols[b, h] = rng.choice(w.N, samples, replace=False)
        out["rows"], out["cols"] = rows, cols
    return out


PATTERNS = ("random", "local", "local_global", "strided", "butterfly")


def block_mask_pattern(pattern, T, rng=None, p=0.125):
    """uint8 [T, T] tile mask (1 = tile computed) of a fixed sparsity pattern.

    The pages define block-sparse attention for any predefined tile mask
    (summary page, "Extension: Block-Sparse FlashAttention") and name none;
    these are common choices:
      random       each tile kept with probability p (draws rng.random((T, T)))
      local        a band: |i - j| <= 2 tiles
      local_global the band |i - j| <= 1 plus tile row 0 and tile column 0
      strided      the band |i - j| <= 1 plus every 8th tile column (j % 8 == 7)
      butterfly    j == i or i XOR j a power of two (the union of the supports
                   of the butterfly factors of a T x T butterfly matrix)
    The diagonal is always kept, so every query row sees at least its own tile."""
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    if pattern == "random":
        m = rng.random((T, T)) < p
    elif pattern == "local":
        m = np.abs(i - j) <= 2
    elif pattern == "local_global":
        m = (np.abs(i - j) <= 1) | (i == 0) | (j == 0)
    elif pattern == "strided":
        m = (np.abs(i - j) <= 1) | (j % 8 == 7)
    elif pattern == "butterfly":
        x = i ^ j
        m = (x & (x - 1)) == 0   # 0 or a single bit
    else:
        raise ValueError("unknown pattern %r" % pattern)
    m = np.array(m, dtype=bool)
    m[np.arange(T), np.arange(T)] = True
    return m.astype(np.uint8)


def random_case(B, H, N, d, seed, dtype="bf16", value_scale=1.0, kv_len=None,
                block_mask=None):
    """Ad-hoc seeded case (edge shapes, ragged tails) with the same recipe."""
    rng = np.random.default_rng(seed)
    out = {}
    for name in ("q", "k", "v", "do"):
        x = rng.standard_normal((B, H, N, d), dtype=np.float32) * np.float32(value_scale)
        if dtype == "bf16":
            out[name], out[name + "_bits"] = bf16_round(x)
        else:
            out[name] = x
    out["kv_len"] = None if kv_len is None else np.asarray(kv_len, np.int32)
    out["block_mask"] = None if block_mask is None else np.asarray(block_mask, np.uint8)
    return out


def sha256(a):
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def flops(w, kept_fraction=None):
    """Algorithmic FLOPs (fwd, fwd+bwd): fwd = 4 B H N^2 d, halved for causal,
    times the kept-tile fraction for block-sparse; bwd = 2.5 x fwd."""
    fwd = 4.0 * w.B * w.H * w.N * w.N * w.d
    if w.causal:
        fwd *= 0.5
    if kept_fraction is not None:
        fwd *= kept_fraction
    return fwd, 3.5 * fwd
