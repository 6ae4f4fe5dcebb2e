"""GPU tests of fused dropout: the keep mask the kernels draw (through both of
their code paths: a query row per thread, a key per thread) equals the oracle's bit for bit, and the forward and
backward with dropout match the fp64 oracle with the same mask within the
bf16 tolerances."""
import numpy as np
import pytest
import torch

import oracle
from oracle import dropout as D
from workloads import random_case
from _gpu_helpers import TOL, f64, max_abs, rel_fro, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("B,H,N,p,seed,offset", [
    (1, 1, 1, 0.5, 0, 0),
    (2, 3, 300, 0.1, 12345, 7),
    (1, 2, 1000, 0.5, 0xDEADBEEF12345678, 0xFFFFFFFF),
    (1, 1, 64, 0.9, 3, 1),
])
def test_mask_bit_exact(fa, path, B, H, N, p, seed, offset):
    # drawn by the kernels' own device code, through the test-only
    # diagnostics library
    import _diag
    out = torch.full((B * H, N, N), 7, dtype=torch.uint8, device="cuda")
    _diag.dropout_mask(out, B, H, N, p, seed, offset, path)
    torch.cuda.synchronize()
    assert _diag.status() == (0, 0)
    got = out.cpu().numpy()
    for bh in range(B * H):
        want = D.keep_mask(np.arange(N), np.arange(N), bh, p, seed, offset)
        assert np.array_equal(got[bh], want.astype(np.uint8)), "head %d" % bh


CASES = [
    # B, H, N, d, causal, mask, p
    (1, 2, 128, 64, False, "none", 0.3),
    (2, 2, 300, 64, True, "none", 0.1),
    (1, 2, 513, 128, False, "none", 0.5),
    (2, 3, 384, 64, False, "padding", 0.2),
    (1, 2, 520, 128, True, "sparse", 0.3),
    (1, 1, 1000, 128, True, "none", 0.9),
    (1, 1, 1, 64, False, "none", 0.5),          # one token
    (2, 2, 200, 128, False, "padding0", 0.3),   # a batch element whose keys are all padding
]


def _case(B, H, N, d, mask, seed):
    rng = np.random.default_rng(seed)
    kv = bm = None
    if mask == "padding":
        kv = rng.integers(1, N + 1, B)
        kv[0] = min(N, 100)
    if mask == "padding0":
        kv = np.array([0] + [N] * (B - 1))
    if mask == "sparse":
        T = (N + 127) // 128
        bm = (rng.random((T, T)) < 0.4).astype(np.uint8)
        bm[np.arange(T), np.arange(T)] = 1
    return random_case(B, H, N, d, seed, kv_len=kv, block_mask=bm)


@pytest.mark.parametrize("B,H,N,d,causal,mask,p", CASES)
def test_dropout_parity(fa, B, H, N, d, causal, mask, p):
    case = _case(B, H, N, d, mask, seed=N + d + int(100 * p))
    t = to_device(case, "bf16")
    seed, offset = 0x5EED0000 + N, 3
    scale = d ** -0.5
    kw = dict(kv_len=t["kv_len"], block_mask=t["block_mask"], dropout_p=p, seed=seed,
              offset=offset)
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, causal, **kw)
    dq, dk, dv = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, causal, **kw)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == 0
    okw = dict(causal=causal, kv_len=case.get("kv_len"), block_mask=case.get("block_mask"),
               dropout=(p, seed, offset))
    ro, rl = oracle.forward(case["q"], case["k"], case["v"], scale, **okw)
    rdq, rdk, rdv, _ = oracle.backward(case["q"], case["k"], case["v"], case["do"], scale, **okw)
    to, tl, tg = TOL["bf16"]
    # O is rescaled by up to 1/(1-p): compare against the tolerance scaled alike
    assert max_abs(f64(o), ro) <= to * D.keep_scale(p), "O"
    assert max_abs(lse.cpu().numpy().astype(np.float64), rl, finite_only=True) <= tl, "lse"
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), (rdq, rdk, rdv)):
        e = rel_fro(f64(g), r)
        assert e <= tg, (name, e)


def test_dropout_determinism_and_offsets(fa):
    B, H, N, d = 1, 2, 384, 64
    case = random_case(B, H, N, d, seed=9)
    t = to_device(case, "bf16")
    run = lambda off: fa.forward(t["q"], t["k"], t["v"], None, True, dropout_p=0.25, seed=11,
                                 offset=off)
    o1, l1 = run(5)
    o2, l2 = run(5)
    o3, l3 = run(6)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(l1, l3)              # lse does not depend on the mask
    assert not torch.equal(o1, o3)          # another offset draws another mask
    # p = 0 through the options is the plain call, bit for bit
    o0, l0 = fa.forward(t["q"], t["k"], t["v"], None, True, dropout_p=0.0, seed=11, offset=5)
    o_plain, l_plain = fa.forward(t["q"], t["k"], t["v"], None, True)
    assert torch.equal(o0, o_plain) and torch.equal(l0, l_plain)


@pytest.mark.slow
def test_dropout_long_causal_sampled(fa):
    """The bench workload's shape with dropout (B 1, H 4, N 16384, d 128,
    causal, p 0.1): 256 sampled query rows per head for O, lse, dQ; the same
    rows as key rows of the first head for dK, dV (the oracle's statistics of
    every row)."""
    B, H, N, d, p, seed, offset = 1, 4, 16384, 128, 0.1, 2024, 1
    case = random_case(B, H, N, d, seed=77, value_scale=0.5)
    t = to_device(case, "bf16")
    scale = d ** -0.5
    kw = dict(dropout_p=p, seed=seed, offset=offset)
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, True, **kw)
    dq, dk, dv = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, True, **kw)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == 0
    rng = np.random.default_rng(78)
    rows = np.stack([np.stack([np.sort(rng.choice(N, 256, replace=False)) for _ in range(H)])])
    drop = (p, seed, offset)
    to, tl, tg = TOL["bf16"]
    take = lambda a, r: np.take_along_axis(a, r[..., None], axis=2)
    ro, rl = oracle.forward_rows(case["q"], case["k"], case["v"], scale, rows, causal=True,
                                 dropout=drop)
    assert max_abs(take(f64(o), rows), ro) <= to * D.keep_scale(p)
    assert max_abs(np.take_along_axis(lse.cpu().numpy().astype(np.float64), rows, axis=2),
                   rl) <= tl
    rdq = oracle.backward_query_rows(case["q"], case["k"], case["v"], case["do"], scale, rows,
                                     causal=True, dropout=drop)
    assert rel_fro(take(f64(dq), rows), rdq) <= tg
    sl = (slice(0, 1), slice(0, 1))
    sub = {n: case[n][sl] for n in ("q", "k", "v", "do")}
    lse_all, d_all = oracle.row_stats(sub["q"], sub["k"], sub["v"], sub["do"], scale,
                                      causal=True, dropout=drop)
    cols = rows[sl]
    rdk, rdv = oracle.backward_key_rows(sub["q"], sub["k"], sub["v"], sub["do"], scale, cols,
                                        lse_all, d_all, causal=True, dropout=drop)
    assert rel_fro(take(f64(dk)[sl], cols), rdk) <= tg
    assert rel_fro(take(f64(dv)[sl], cols), rdv) <= tg
