"""Plain fp64 CPU oracle for exact (masked, scaled) softmax attention.

TEST INFRASTRUCTURE ONLY: imported by `tests/`, `__graft_entry__.smoke()` and
the CPU-baseline leg of `bench.py`, never by the product path.

What it computes is the plain definition of attention, because the tiled method
reaches that exact result up to floating-point rounding ("FlashAttention: Fast
and Memory-Efficient Exact Attention with IO-Awareness", summary page, sections
"Problem and motivation" and Q&A: exact attention, same output).  For one
(batch, head) slice with query rows q_i, key rows k_j and value rows v_j:

    S_ij = scale * q_i . k_j          if key j is visible from query i, else -inf
    m_i  = max_j S_ij
    P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i)           (safe softmax)
    O_i  = sum_j P_ij v_j
    lse_i = m_i + ln sum_j exp(S_ij - m_i)

Sources for each piece:
  * S = Q K^T, P = softmax(S), O = P V -- the FlashAttention summary page,
    "Problem and motivation"; also "From Online Softmax to FlashAttention"
    (blog review), section "The Self-Attention".
  * the scale applied to the scores -- GitHub issue "Fewer matrix
    multiplications, same results" (flash-attention #941), where the query
    block is multiplied by 1/sqrt(d) before the Q K^T product.
  * subtracting the row maximum -- blog review, section "(safe) softmax".
  * keeping only (m, l) (here folded into lse = m + ln l) for the backward --
    summary page, "Key ideas: recomputation in the backward pass".
  * masking -- glossary page "Flash Attention", "Normalization and Masking";
    causal keeps j <= i (GitHub issue, lower-triangular mask); block-sparse
    keeps a tile (i//B, j//B) only where the tile mask is 1 (summary page,
    "Extension: block-sparse FlashAttention").

The backward pass is not written out on any of the pages (they only say that
S and P are recomputed from Q, K and the saved statistics).  Its formulas here
are the textbook derivative of L(O) through the definition above:

    dV = P^T dO,   dP = dO V^T,   D_i = sum_j P_ij dP_ij,
    dS = P o (dP - D),   dQ = scale * dS K,   dK = scale * dS^T Q.

Readings taken where the pages are silent:
  * a query row with no visible key has O_i = 0, lse_i = -inf and contributes
    no gradient;
  * key padding masks keys j >= kv_len[b] only; padded query rows are computed
    normally;
  * the block-sparse tile mask is one T x T 0/1 array shared by every (b, h),
    T = ceil(N / block).

An additive score bias (optional argument `bias`, any array broadcastable to
[B, H, N, N]: the "+ mask" term of the score definition taken as a tensor) is
added to the scaled scores before the masks: S_ij = scale q_i . k_j + bias_ij;
bias entries of -inf hide a key like a mask.

Dropout (optional argument `dropout=(p, seed, offset)` of the whole-tensor and
sampled-row functions) follows `oracle/dropout.py`: O = (P o Z) V / (1 - p)
with the mask Z of that module, and the chain rule through it.

Rows of the score matrix are independent by definition, so functions that
handle long sequences evaluate whole rows a group of rows at a time; nothing
else is blocked, fused or reordered.  All arithmetic is float64 on inputs that
the caller has already rounded to the precision the GPU sees.
"""
import numpy as np

from . import dropout as _dropout

__all__ = [
    "visible", "scores", "probabilities", "forward", "backward",
    "forward_rows", "backward_query_rows", "backward_key_rows", "row_stats",
    "softmax_three_pass", "softmax_online_two_pass",
    "attention_row_one_pass_tiled", "row_block_forward_backward",
]


# --------------------------------------------------------------------------
# masks
# --------------------------------------------------------------------------

def visible(rows, n_keys, causal=False, kv_len_b=None, block_mask=None, block=128, keys=None):
    """Boolean visibility of keys 0..n_keys-1 (or of the key indices `keys`)
    from the given query rows.

    rows      : 1-D integer array of query indices (or an int N for 0..N-1)
    causal    : keep j <= i (lower-triangular mask, GitHub issue #941)
    kv_len_b  : keep j < kv_len_b (key padding of one batch element)
    block_mask: T x T array of 0/1; keep (i, j) where block_mask[i//block][j//block]
    """
    if np.isscalar(rows):
        rows = np.arange(int(rows))
    rows = np.asarray(rows, dtype=np.int64)
    cols = (np.arange(n_keys, dtype=np.int64) if keys is None
            else np.asarray(keys, dtype=np.int64))
    vis = np.ones((rows.size, cols.size), dtype=bool)
    if causal:
        vis &= cols[None, :] <= rows[:, None]
    if kv_len_b is not None:
        vis &= cols[None, :] < int(kv_len_b)
    if block_mask is not None:
        bm = np.asarray(block_mask).astype(bool)
        vis &= bm[rows[:, None] // block, cols[None, :] // block]
    return vis


def _kv_len_of(kv_len, b):
    return None if kv_len is None else int(np.asarray(kv_len)[b])


# --------------------------------------------------------------------------
# the definition, one (b, h) slice at a time
# --------------------------------------------------------------------------

def scores(q, k, scale, vis, bias=None):
    """S = scale * q k^T (+ bias [R,N]) with -inf where a key is not visible.
    q: [R,d], k: [N,d]."""
    s = scale * (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T)
    if bias is not None:
        s = s + np.asarray(bias, np.float64)
    return np.where(vis, s, -np.inf)


def _bias_of(bias, b, h):
    """The [N, N] bias of slice (b, h) (broadcast over size-1 leading axes)."""
    if bias is None:
        return None
    bias = np.asarray(bias)
    return bias[b if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0]


def _rows(x, r):
    return None if x is None else x[r]


def probabilities(s):
    """Safe softmax of each row of s (blog review, "(safe) softmax").

    Returns (P, lse).  A row whose entries are all -inf gets P = 0 and
    lse = -inf.
    """
    m = np.max(s, axis=1, keepdims=True)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe)  # exp(-inf) = 0 for masked entries
    l = np.sum(e, axis=1, keepdims=True)
    l_safe = np.where(empty, 1.0, l)
    p = np.where(empty, 0.0, e / l_safe)
    with np.errstate(divide="ignore"):
        lse = np.where(empty[:, 0], -np.inf, m_safe[:, 0] + np.log(l_safe[:, 0]))
    return p, lse


def _drop(dropout, rows, cols, bh):
    """(Z, scale) of the dropout mask for query `rows` x key `cols` of head
    bh, or (None, 1) without dropout."""
    if dropout is None or _dropout.threshold(dropout[0]) == 0:
        return None, 1.0
    p, seed, offset = dropout
    return _dropout.keep_mask(rows, cols, bh, p, seed, offset), _dropout.keep_scale(p)


def _slice_forward(q, k, v, scale, vis, z=None, rp=1.0, bias=None):
    p, lse = probabilities(scores(q, k, scale, vis, bias))
    pd = p if z is None else p * z * rp
    return pd @ np.asarray(v, np.float64), lse, p


def _slice_backward(q, k, v, do, scale, vis, z=None, rp=1.0, bias=None):
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    p, _ = probabilities(scores(q, k, scale, vis, bias))
    pd = p if z is None else p * z * rp
    dv = pd.T @ do
    dp = do @ v.T
    if z is not None:
        dp = dp * z * rp
    d_row = np.sum(p * dp, axis=1)
    ds = p * (dp - d_row[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, d_row


# --------------------------------------------------------------------------
# whole tensors [B, H, N, d]
# --------------------------------------------------------------------------

def forward(q, k, v, scale, causal=False, kv_len=None, block_mask=None, block=128,
            dropout=None, bias=None):
    """O [B,H,N,d] and lse [B,H,N] (natural log) for q, k, v of shape [B,H,N,d]."""
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, d), np.float64)
    lse = np.zeros((B, H, N), np.float64)
    for b in range(B):
        vis = visible(N, k.shape[2], causal, _kv_len_of(kv_len, b), block_mask, block)
        for h in range(H):
            z, rp = _drop(dropout, np.arange(N), np.arange(k.shape[2]), b * H + h)
            o[b, h], lse[b, h], _ = _slice_forward(q[b, h], k[b, h], v[b, h], scale, vis, z, rp,
                                                   _bias_of(bias, b, h))
    return o, lse


def backward(q, k, v, do, scale, causal=False, kv_len=None, block_mask=None, block=128,
             dropout=None, bias=None):
    """(dQ, dK, dV, D) for the loss sum(O * dO); D [B,H,N] = rowsum(P o dP)."""
    B, H, N, d = q.shape
    dq = np.zeros((B, H, N, d), np.float64)
    dk = np.zeros_like(dq)
    dv = np.zeros_like(dq)
    dd = np.zeros((B, H, N), np.float64)
    for b in range(B):
        vis = visible(N, k.shape[2], causal, _kv_len_of(kv_len, b), block_mask, block)
        for h in range(H):
            z, rp = _drop(dropout, np.arange(N), np.arange(k.shape[2]), b * H + h)
            dq[b, h], dk[b, h], dv[b, h], dd[b, h] = _slice_backward(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, vis, z, rp, _bias_of(bias, b, h))
    return dq, dk, dv, dd


# --------------------------------------------------------------------------
# sampled rows, for sequences too long to check every output
# --------------------------------------------------------------------------

def forward_rows(q, k, v, scale, rows, causal=False, kv_len=None, block_mask=None,
                 block=128, dropout=None, bias=None):
    """O and lse of the selected query rows; rows: int array [B,H,R]."""
    B, H, N, d = q.shape
    R = rows.shape[2]
    o = np.zeros((B, H, R, d), np.float64)
    lse = np.zeros((B, H, R), np.float64)
    for b in range(B):
        for h in range(H):
            vis = visible(rows[b, h], N, causal, _kv_len_of(kv_len, b), block_mask, block)
            z, rp = _drop(dropout, rows[b, h], np.arange(N), b * H + h)
            o[b, h], lse[b, h], _ = _slice_forward(q[b, h][rows[b, h]], k[b, h],
                                                   v[b, h], scale, vis, z, rp,
                                                   _rows(_bias_of(bias, b, h), rows[b, h]))
    return o, lse


def backward_query_rows(q, k, v, do, scale, rows, causal=False, kv_len=None,
                        block_mask=None, block=128, dropout=None, bias=None):
    """dQ of the selected query rows.  Everything dQ_i needs is in row i:
    P_i., dP_i. = dO_i V^T, D_i = sum_j P_ij dP_ij."""
    B, H, N, d = q.shape
    R = rows.shape[2]
    dq = np.zeros((B, H, R, d), np.float64)
    for b in range(B):
        for h in range(H):
            r = rows[b, h]
            vis = visible(r, N, causal, _kv_len_of(kv_len, b), block_mask, block)
            p, _ = probabilities(scores(q[b, h][r], k[b, h], scale, vis,
                                        _rows(_bias_of(bias, b, h), r)))
            dp = np.asarray(do[b, h][r], np.float64) @ np.asarray(v[b, h], np.float64).T
            z, rp = _drop(dropout, r, np.arange(N), b * H + h)
            if z is not None:
                dp = dp * z * rp
            d_row = np.sum(p * dp, axis=1)
            ds = p * (dp - d_row[:, None])
            dq[b, h] = scale * (ds @ np.asarray(k[b, h], np.float64))
    return dq


def row_stats(q, k, v, do, scale, causal=False, kv_len=None, block_mask=None,
              block=128, rows_per_group=1024, dropout=None, bias=None):
    """lse_i and D_i = sum_j P_ij dP_ij for EVERY query row, [B,H,N] each.

    Rows are taken a group at a time so that the score rows of a long
    sequence need not all be held at once."""
    B, H, N, d = q.shape
    lse = np.zeros((B, H, N), np.float64)
    dd = np.zeros((B, H, N), np.float64)
    for b in range(B):
        for h in range(H):
            kf = np.asarray(k[b, h], np.float64)
            vf = np.asarray(v[b, h], np.float64)
            for r0 in range(0, N, rows_per_group):
                r = np.arange(r0, min(N, r0 + rows_per_group))
                vis = visible(r, N, causal, _kv_len_of(kv_len, b), block_mask, block)
                p, lse[b, h, r] = probabilities(scores(q[b, h][r], kf, scale, vis,
                                                       _rows(_bias_of(bias, b, h), r)))
                dp = np.asarray(do[b, h][r], np.float64) @ vf.T
                z, rp = _drop(dropout, r, np.arange(N), b * H + h)
                if z is not None:
                    dp = dp * z * rp
                dd[b, h, r] = np.sum(p * dp, axis=1)
    return lse, dd


def backward_key_rows(q, k, v, do, scale, cols, lse, dd, causal=False, kv_len=None,
                      block_mask=None, block=128, dropout=None, bias=None):
    """dK and dV of the selected key rows (cols: int array [B,H,C]).

    dK_j and dV_j sum over every query row, so they need every row's lse and
    D (from `row_stats`):  P_ij = exp(S_ij - lse_i),  dS_ij = P_ij (dP_ij - D_i),
    dV_j = sum_i P_ij dO_i,  dK_j = scale * sum_i dS_ij q_i."""
    B, H, N, d = q.shape
    C = cols.shape[2]
    dk = np.zeros((B, H, C, d), np.float64)
    dv = np.zeros((B, H, C, d), np.float64)
    rows = np.arange(N)
    for b in range(B):
        for h in range(H):
            c = cols[b, h]
            qf = np.asarray(q[b, h], np.float64)
            dof = np.asarray(do[b, h], np.float64)
            vis = visible(rows, N, causal, _kv_len_of(kv_len, b), block_mask, block, keys=c)
            bb = _bias_of(bias, b, h)
            s = scores(qf, k[b, h][c], scale, vis, None if bb is None else bb[:, c])  # [N, C]
            l = lse[b, h][:, None]
            with np.errstate(invalid="ignore"):
                p = np.where(vis & np.isfinite(l), np.exp(s - np.where(np.isfinite(l), l, 0.0)), 0.0)
            dp = dof @ np.asarray(v[b, h][c], np.float64).T         # [N, C]
            z, rp = _drop(dropout, rows, c, b * H + h)
            pd = p
            if z is not None:
                dp = dp * z * rp
                pd = p * z * rp
            ds = p * (dp - dd[b, h][:, None])
            dv[b, h] = pd.T @ dof
            dk[b, h] = scale * (ds.T @ qf)
    return dk, dv


def row_block_forward_backward(q, k, v, do, scale, b, h, rows, causal=False, kv_len=None,
                               block_mask=None, block=128):
    """Forward and backward of one block of query rows of slice (b, h), the
    definition restricted to those rows: O, lse and dQ of the rows, and the
    rows' contributions P^T dO and scale dS^T Q to dV and dK.  Summing the
    contributions of every row block gives the full dK, dV."""
    r = np.asarray(rows, np.int64)
    N = k.shape[2]
    vis = visible(r, N, causal, _kv_len_of(kv_len, b), block_mask, block)
    qf = np.asarray(q[b, h][r], np.float64)
    kf = np.asarray(k[b, h], np.float64)
    vf = np.asarray(v[b, h], np.float64)
    dof = np.asarray(do[b, h][r], np.float64)
    p, lse = probabilities(scores(qf, kf, scale, vis))
    o = p @ vf
    dp = dof @ vf.T
    d_row = np.sum(p * dp, axis=1)
    ds = p * (dp - d_row[:, None])
    dq = scale * (ds @ kf)
    dk_part = scale * (ds.T @ qf)
    dv_part = p.T @ dof
    return o, lse, dq, dk_part, dv_part


# --------------------------------------------------------------------------
# the derivation chain of the blog review "From Online Softmax to
# FlashAttention", used to pin the oracle's definition against the
# recurrences that the tiled kernels implement
# --------------------------------------------------------------------------

def softmax_three_pass(x):
    """Section "(safe) softmax", 3-pass algorithm: a running max m_i over the
    whole vector, then d_i = d_{i-1} + exp(x_i - m_N), then a_i = exp(x_i - m_N)/d_N."""
    x = np.asarray(x, np.float64)
    m = -np.inf
    for xi in x:
        m = max(m, xi)
    d = 0.0
    for xi in x:
        d = d + np.exp(xi - m)
    return np.array([np.exp(xi - m) / d for xi in x]), m, d


def softmax_online_two_pass(x):
    """Section "Online Softmax", 2-pass algorithm: in one pass
    m_i = max(m_{i-1}, x_i) and d'_i = d'_{i-1} exp(m_{i-1} - m_i) + exp(x_i - m_i);
    then a_i = exp(x_i - m_N) / d'_N."""
    x = np.asarray(x, np.float64)
    m_prev, d_prev = -np.inf, 0.0
    for xi in x:
        m_i = max(m_prev, xi)
        scale_prev = 0.0 if m_prev == -np.inf else np.exp(m_prev - m_i)
        d_prev = d_prev * scale_prev + np.exp(xi - m_i)
        m_prev = m_i
    return np.array([np.exp(xi - m_prev) / d_prev for xi in x]), m_prev, d_prev


def attention_row_one_pass_tiled(x, v, tile_starts):
    """Section "Algorithm FlashAttention (Tiling)" for one query row.

    x: the row's pre-softmax logits [N]; v: value rows [N, d]; tile_starts:
    increasing start indices of the key tiles (first 0).  Per tile t:
    local max, m_t = max(m_{t-1}, local max),
    d'_t = d'_{t-1} exp(m_{t-1} - m_t) + sum_j exp(x_j - m_t),
    o'_t = o'_{t-1} d'_{t-1} exp(m_{t-1} - m_t) / d'_t + sum_j exp(x_j - m_t)/d'_t v_j.
    Returns (o'_last, m_last, d'_last)."""
    x = np.asarray(x, np.float64)
    v = np.asarray(v, np.float64)
    bounds = list(tile_starts) + [x.size]
    m_prev, d_prev = -np.inf, 0.0
    o_prev = np.zeros(v.shape[1], np.float64)
    for t in range(len(bounds) - 1):
        xs = x[bounds[t]:bounds[t + 1]]
        vs = v[bounds[t]:bounds[t + 1]]
        m_local = np.max(xs)
        m_t = max(m_prev, m_local)
        carry = 0.0 if m_prev == -np.inf else np.exp(m_prev - m_t)
        e = np.exp(xs - m_t)
        d_t = d_prev * carry + np.sum(e)
        o_prev = o_prev * (d_prev * carry / d_t) + (e / d_t) @ vs
        m_prev, d_prev = m_t, d_t
    return o_prev, m_prev, d_prev
