"""Dropout on the attention probabilities, fp64 CPU oracle -- TEST
INFRASTRUCTURE ONLY (imported by `tests/`, never by the product path).

The pages list dropout among the operations the kernel fuses with the matrix
products, the mask and the softmax, and say that the backward pass keeps the
state of the pseudo-random generator to regenerate the dropout mask on chip
instead of storing it (summary page "FlashAttention: Fast and Memory-Efficient
Exact Attention with IO-Awareness", "Key ideas: kernel fusion" and the question
on the auxiliary memory of the backward pass).  They fix neither where the
dropout acts nor the generator.  Readings taken here:

  * Dropout acts on the attention probabilities, as in the usual attention
    layer: with Z_ij in {0, 1} drawn independently, keep probability 1 - p,
        O = (P o Z) V / (1 - p)
    and lse is that of the undropped scores.
  * The backward is the chain rule through that definition:
        dV = (P o Z)^T dO / (1 - p),   dP = (dO V^T) o Z / (1 - p),
        D_i = sum_j P_ij dP_ij  (= dO_i . O_i),   dS = P o (dP - D),
        dQ = scale dS K,   dK = scale dS^T Q.
  * Generator: Philox4x32-10, the counter-based generator of Salmon, Moraes,
    Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC 2011),
    written from its published definition: a 4 x 32-bit counter, a 2 x 32-bit
    key, ten rounds; each round multiplies counter words 0 and 2 by the
    constants M0 = 0xD2511F53 and M1 = 0xCD9E8D57 into 64-bit products and
    maps (c0, c1, c2, c3) to (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
    lo(M0 c0)); between rounds the key is bumped by the Weyl constants
    W0 = 0x9E3779B9, W1 = 0xBB67AE85.
  * Counter layout (this library's choice): the element (i, j) of head
    (b, h) uses the call with counter (j // 8, i, b*H + h, offset) and key
    (seed mod 2^32, seed div 2^32); its four output words hold eight 16-bit
    uniforms, key j taking the low (j even) or high (j odd) half of word
    (j mod 8) // 2.  Z_ij = 1 (kept) iff that uniform is >= t, where
    t = min(65535, floor(p 65536 + 1/2)) with p rounded to float32 first, so
    the keep probability is exactly 1 - t/65536 and the scale is
    65536 / (65536 - t).
"""
import numpy as np

__all__ = ["PHILOX_M0", "PHILOX_M1", "PHILOX_W0", "PHILOX_W1", "philox4x32_10",
           "philox4x32_10_scalar", "threshold", "keep_scale", "keep_mask"]

PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85
_MASK32 = 0xFFFFFFFF


def philox4x32_10_scalar(ctr, key):
    """Philox4x32-10 on Python integers: ctr (c0, c1, c2, c3), key (k0, k1)."""
    c0, c1, c2, c3 = (int(x) & _MASK32 for x in ctr)
    k0, k1 = (int(x) & _MASK32 for x in key)
    for _ in range(10):
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0, p1 & _MASK32, (p0 >> 32) ^ c3 ^ k1,
                          p0 & _MASK32)
        k0 = (k0 + PHILOX_W0) & _MASK32
        k1 = (k1 + PHILOX_W1) & _MASK32
    return c0, c1, c2, c3


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """The same on numpy arrays (broadcast), as uint64 holding 32-bit values."""
    u = np.uint64
    c0, c1, c2, c3 = (np.asarray(x, np.uint64) & u(_MASK32) for x in (c0, c1, c2, c3))
    k0 = u(int(k0) & _MASK32)
    k1 = u(int(k1) & _MASK32)
    m32 = u(_MASK32)
    for _ in range(10):
        p0 = c0 * u(PHILOX_M0)          # < 2^64: exact in uint64
        p1 = c2 * u(PHILOX_M1)
        c0, c1, c2, c3 = ((p1 >> u(32)) ^ c1 ^ k0, p1 & m32, (p0 >> u(32)) ^ c3 ^ k1,
                          p0 & m32)
        k0 = (k0 + u(PHILOX_W0)) & m32
        k1 = (k1 + u(PHILOX_W1)) & m32
    return c0, c1, c2, c3


def threshold(p):
    """The 16-bit drop threshold t of probability p (p rounded to float32)."""
    p32 = float(np.float32(p))
    if not 0.0 <= p32 < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return min(65535, int(np.floor(p32 * 65536.0 + 0.5)))


def keep_scale(p):
    """1 / (1 - t/65536), the factor applied to the kept probabilities."""
    t = threshold(p)
    return 65536.0 / (65536.0 - t)


def keep_mask(rows, cols, bh, p, seed, offset):
    """Z[r, c] (bool) for query indices `rows` and key indices `cols` of head
    bh = b*H + h."""
    rows = np.asarray(rows, np.int64)
    cols = np.asarray(cols, np.int64)
    t = threshold(p)
    if t == 0:
        return np.ones((rows.size, cols.size), bool)
    groups, inv = np.unique(cols >> 3, return_inverse=True)
    w = philox4x32_10(groups[None, :], rows[:, None], bh, offset, seed & _MASK32,
                      (seed >> 32) & _MASK32)
    words = np.stack(np.broadcast_arrays(*w), axis=-1)[:, inv, :]   # [R, C, 4]
    sel = ((cols & 7) >> 1)[None, :, None]
    word = np.take_along_axis(words, np.broadcast_to(sel, (rows.size, cols.size, 1)),
                              axis=2)[..., 0]
    half = (cols & 1).astype(np.uint64)[None, :] * np.uint64(16)
    u16 = (word >> half) & np.uint64(0xFFFF)
    return u16 >= np.uint64(t)
