"""GPU tests of the additive score bias: against the fp64 oracle with the
same bias (full, broadcast over batch and/or heads, with hidden keys, combined
with the masks and with dropout) within the bf16 tolerances."""
import numpy as np
import pytest
import torch

import oracle
from oracle import dropout as D
from workloads import random_case
from _gpu_helpers import TOL, f64, max_abs, rel_fro, to_device

pytestmark = pytest.mark.gpu


def run_case(fa, case, bias_np, B, H, N, d, causal, drop=None):
    t = to_device(case, "bf16")
    # rows padded to a multiple of 4 floats (the 16-byte row-stride rule)
    N4 = (N + 3) // 4 * 4
    padded = torch.zeros(bias_np.shape[:3] + (N4,), dtype=torch.float32, device="cuda")
    padded[..., :N] = torch.from_numpy(np.ascontiguousarray(bias_np, dtype=np.float32)).cuda()
    bias = padded[..., :N]
    scale = d ** -0.5
    kw = dict(kv_len=t["kv_len"], block_mask=t["block_mask"], bias=bias)
    if drop:
        kw.update(dropout_p=drop[0], seed=drop[1], offset=drop[2])
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, causal, **kw)
    dq, dk, dv = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, causal, **kw)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == 0
    okw = dict(causal=causal, kv_len=case.get("kv_len"), block_mask=case.get("block_mask"),
               bias=bias_np.astype(np.float64), dropout=drop)
    ro, rl = oracle.forward(case["q"], case["k"], case["v"], scale, **okw)
    rdq, rdk, rdv, _ = oracle.backward(case["q"], case["k"], case["v"], case["do"], scale, **okw)
    to, tl, tg = TOL["bf16"]
    rp = D.keep_scale(drop[0]) if drop else 1.0
    lse_np = lse.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(lse_np), np.isneginf(rl)), "empty-row pattern"
    assert max_abs(f64(o), ro) <= to * rp, "O"
    assert max_abs(lse_np, rl, finite_only=True) <= tl, "lse"
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), (rdq, rdk, rdv)):
        e = rel_fro(f64(g), r)
        assert e <= tg, (name, e)


def _mask_args(B, N, mask, rng):
    kv = bm = None
    if mask == "padding":
        kv = rng.integers(1, N + 1, B)
    if mask == "sparse":
        T = (N + 127) // 128
        bm = (rng.random((T, T)) < 0.4).astype(np.uint8)
        bm[np.arange(T), np.arange(T)] = 1
    return kv, bm


@pytest.mark.parametrize("B,H,N,d,causal,mask,shape", [
    (1, 2, 128, 64, False, "none", "full"),
    (2, 2, 300, 64, True, "none", "full"),
    (1, 2, 513, 128, False, "none", "one"),       # one [N, N] bias for every head
    (2, 3, 384, 64, False, "padding", "heads"),   # per head, broadcast over batch
    (2, 2, 520, 128, True, "sparse", "batch"),    # per batch element, broadcast over heads
    (1, 1, 1, 64, False, "none", "full"),
])
def test_bias_parity(fa, B, H, N, d, causal, mask, shape):
    rng = np.random.default_rng(N + d)
    kv, bm = _mask_args(B, N, mask, rng)
    case = random_case(B, H, N, d, seed=N + 3 * d, kv_len=kv, block_mask=bm)
    dims = {"full": (B, H), "one": (1, 1), "heads": (1, H), "batch": (B, 1)}[shape]
    bias = rng.standard_normal(dims + (N, N)).astype(np.float32)
    run_case(fa, case, bias, B, H, N, d, causal)


def test_bias_hidden_keys_and_empty_rows(fa):
    """-inf entries hide keys; rows hidden entirely give O = 0, lse = -inf."""
    B, H, N, d = 1, 2, 260, 128
    rng = np.random.default_rng(5)
    case = random_case(B, H, N, d, seed=6)
    bias = rng.standard_normal((B, H, N, N)).astype(np.float32)
    bias[rng.random(bias.shape) < 0.3] = -np.inf
    bias[:, :, [0, 100, 259], :] = -np.inf   # three rows with no visible key
    run_case(fa, case, bias, B, H, N, d, False)


def test_bias_with_dropout(fa):
    B, H, N, d = 2, 2, 384, 64
    rng = np.random.default_rng(7)
    case = random_case(B, H, N, d, seed=8)
    bias = (rng.standard_normal((1, H, N, N)) * 2).astype(np.float32)
    run_case(fa, case, bias, B, H, N, d, True, drop=(0.2, 99, 4))


def test_causal_bias_equals_causal_mask(fa):
    """A -inf upper triangle as a bias gives the causal result (through the
    other kernel variant), to within rounding."""
    B, H, N, d = 1, 2, 300, 64
    case = random_case(B, H, N, d, seed=9)
    t = to_device(case, "bf16")
    i, j = np.indices((N, N))
    bias = torch.from_numpy(np.where(j > i, -np.inf, 0.0).astype(np.float32)[None, None]).cuda()
    o0, l0 = fa.forward(t["q"], t["k"], t["v"], None, True)
    o1, l1 = fa.forward(t["q"], t["k"], t["v"], None, False, bias=bias)
    g0 = fa.backward(t["q"], t["k"], t["v"], o0, t["do"], l0, None, True)
    g1 = fa.backward(t["q"], t["k"], t["v"], o1, t["do"], l1, None, False, bias=bias)
    torch.cuda.synchronize()
    assert max_abs(f64(o0), f64(o1)) <= 1e-2
    assert max_abs(l0.cpu().numpy().astype(np.float64), l1.cpu().numpy().astype(np.float64)) <= 1e-4
    for a, b in zip(g0, g1):
        assert rel_fro(f64(b), f64(a)) <= 1e-2


def test_everything_together(fa):
    """[B,N,H,d] inputs and outputs, a padded-row dO, dropout, a per-head bias,
    causal and key padding in one call, against the oracle on dense arrays."""
    B, H, N, d = 2, 3, 333, 128
    rng = np.random.default_rng(12)
    kv = rng.integers(100, N + 1, B)
    case = random_case(B, H, N, d, seed=13, kv_len=kv)
    t = to_device(case, "bf16")
    bnhd = lambda x: x.transpose(1, 2).contiguous().transpose(1, 2)   # [B,N,H,d] storage
    q, k, v = bnhd(t["q"]), bnhd(t["k"]), bnhd(t["v"])
    do_buf = torch.zeros(B, H, N, d + 64, dtype=torch.bfloat16, device="cuda")
    do_buf[..., :d] = t["do"]
    do = do_buf[..., :d]
    N4 = (N + 3) // 4 * 4
    bias_np = rng.standard_normal((1, H, N, N)).astype(np.float32)
    bias_buf = torch.zeros(1, H, N, N4, dtype=torch.float32, device="cuda")
    bias_buf[..., :N] = torch.from_numpy(bias_np).cuda()
    bias = bias_buf[..., :N]
    drop = (0.15, 4242, 17)
    kw = dict(kv_len=t["kv_len"], bias=bias, dropout_p=drop[0], seed=drop[1], offset=drop[2])
    scale = d ** -0.5
    o, lse = fa.forward(q, k, v, scale, True, **kw)
    assert o.stride() == q.stride()
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, scale, True, **kw)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == 0
    okw = dict(causal=True, kv_len=case["kv_len"], bias=bias_np.astype(np.float64), dropout=drop)
    ro, rl = oracle.forward(case["q"], case["k"], case["v"], scale, **okw)
    rdq, rdk, rdv, _ = oracle.backward(case["q"], case["k"], case["v"], case["do"], scale, **okw)
    to, tl, tg = TOL["bf16"]
    assert max_abs(f64(o), ro) <= to * D.keep_scale(drop[0])
    assert max_abs(lse.cpu().numpy().astype(np.float64), rl, finite_only=True) <= tl
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), (rdq, rdk, rdv)):
        assert rel_fro(f64(g), r) <= tg, name


def test_everything_together_d64(fa):
    """The d = 64 kernels with every option at once, as the test above does for
    d = 128: Q, K, V, dO (and so O and the gradients) as [B, N, H, d] buffers
    seen through [B, H, N, d] views, a per-head bias, dropout, the causal mask
    and key padding, against the oracle on the same values."""
    B, H, N, d, p, seed, offset = 2, 3, 300, 64, 0.2, 4242, 9
    rng = np.random.default_rng(77)
    kv = rng.integers(1, N + 1, B)
    case = random_case(B, H, N, d, seed=78, kv_len=kv)
    t = to_device(case, "bf16")
    views = {}
    for n in ("q", "k", "v", "do"):
        buf = torch.empty((B, N, H, d), dtype=torch.bfloat16, device="cuda")
        views[n] = buf.transpose(1, 2)
        views[n].copy_(t[n])
    bias_np = rng.standard_normal((1, H, N, N)).astype(np.float32)
    bias = torch.from_numpy(bias_np).cuda()
    scale = d ** -0.5
    kw = dict(kv_len=t["kv_len"], bias=bias, dropout_p=p, seed=seed, offset=offset)
    o, lse = fa.forward(views["q"], views["k"], views["v"], scale, True, **kw)
    assert o.stride() == views["q"].stride()
    dq, dk, dv = fa.backward(views["q"], views["k"], views["v"], o, views["do"], lse, scale,
                             True, **kw)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == 0
    okw = dict(causal=True, kv_len=kv, bias=bias_np.astype(np.float64),
               dropout=(p, seed, offset))
    ro, rl = oracle.forward(case["q"], case["k"], case["v"], scale, **okw)
    rdq, rdk, rdv, _ = oracle.backward(case["q"], case["k"], case["v"], case["do"], scale, **okw)
    to, tl, tg = TOL["bf16"]
    assert max_abs(f64(o), ro) <= to * D.keep_scale(p), "O"
    assert max_abs(lse.cpu().numpy().astype(np.float64), rl, finite_only=True) <= tl, "lse"
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), (rdq, rdk, rdv)):
        e = rel_fro(f64(g), r)
        assert e <= tg, (name, e)
