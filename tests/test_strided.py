"""GPU tests of the *_ex calls with layouts: the same values laid out in other
layouts ([B,N,H,d], a slot of a packed QKV buffer, padded rows, heads
outermost) must give bit for bit the results of the dense call, the outputs
written through their own strides and nothing outside their views touched.
One case is also compared with the fp64 oracle directly."""
import numpy as np
import pytest
import torch

import oracle
from workloads import random_case
from _gpu_helpers import TOL, f64, max_abs, rel_fro, to_device

pytestmark = pytest.mark.gpu

FILL = -7.0  # sentinel, exact in bf16 and fp32
KINDS = ("dense", "bnhd", "packed", "padded", "hbnd")


def place(shape, dtype, kind, x=None):
    """(buffer, [B,H,N,d] view of it in layout `kind`), the buffer filled with
    FILL and the view with x when given."""
    B, H, N, d = shape
    full = lambda *s: torch.full(s, FILL, dtype=dtype, device="cuda")
    if kind == "dense":
        buf = full(B, H, N, d)
        view = buf
    elif kind == "bnhd":      # heads side by side in each token's row
        buf = full(B, N, H, d)
        view = buf.transpose(1, 2)
    elif kind == "packed":    # slot 1 of a [B, N, 3, H, d] QKV projection
        buf = full(B, N, 3, H, d)
        view = buf[:, :, 1].transpose(1, 2)
    elif kind == "padded":    # rows of d + 64 elements
        buf = full(B, H, N, d + 64)
        view = buf[..., :d]
    elif kind == "hbnd":      # heads outermost
        buf = full(H, B, N, d)
        view = buf.transpose(0, 1)
    else:
        raise ValueError(kind)
    if x is not None:
        view.copy_(x)
    return buf, view


def untouched_outside(buf, kind, shape):
    """True when every element of buf outside the view still holds FILL."""
    mask_buf, mask_view = place(shape, torch.float32, kind)
    mask_buf.fill_(1.0)
    mask_view.fill_(0.0)
    outside = mask_buf.bool()
    return bool((buf[outside].float() == FILL).all())


def run_dense(fa, t, B, H, N, d, scale, causal, mask, fp32):
    o = torch.empty_like(t["q"])
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    (fa.fa_fwd_fp32 if fp32 else fa.fa_fwd)(t["q"], t["k"], t["v"], o, lse, B, H, N, d, scale,
                                            causal, mask)
    dq, dk, dv = (torch.empty_like(t["q"]) for _ in range(3))
    ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    (fa.fa_bwd_fp32 if fp32 else fa.fa_bwd)(t["q"], t["k"], t["v"], o, t["do"], lse, dq, dk, dv,
                                            ws, ws_bytes, B, H, N, d, scale, causal, mask)
    return o, lse, dq, dk, dv


def run_strided(fa, t, shape, scale, causal, mask, fp32, kinds):
    """kinds: layout per tensor name (q, k, v, o, dO, dq, dk, dv)."""
    B, H, N, d = shape
    dt = t["q"].dtype
    bufs, views = {}, {}
    for name, src in (("q", t["q"]), ("k", t["k"]), ("v", t["v"]), ("dO", t["do"])):
        bufs[name], views[name] = place(shape, dt, kinds[name], src)
    for name in ("o", "dq", "dk", "dv"):
        bufs[name], views[name] = place(shape, dt, kinds[name])
    lse = torch.full((B, H, N), FILL, dtype=torch.float32, device="cuda")
    opt = fa.make_options(fa.make_layouts(**views))
    (fa.fa_fwd_fp32_ex if fp32 else fa.fa_fwd_ex)(
        views["q"], views["k"], views["v"], views["o"], lse, B, H, N, d, scale, causal, mask,
        opt)
    ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    (fa.fa_bwd_fp32_ex if fp32 else fa.fa_bwd_ex)(
        views["q"], views["k"], views["v"], views["o"], views["dO"], lse, views["dq"],
        views["dk"], views["dv"], ws, ws_bytes, B, H, N, d, scale, causal, mask, opt)
    torch.cuda.synchronize()
    code, site = fa.fa_get_device_status()
    assert code == 0, "device status %d at site %d" % (code, site)
    for name in ("o", "dq", "dk", "dv"):
        assert untouched_outside(bufs[name], kinds[name], shape), name + " wrote outside its view"
    return views["o"], lse, views["dq"], views["dk"], views["dv"]


def make_case(B, H, N, d, mask_kind, seed, dtype):
    rng = np.random.default_rng(seed)
    kv = bm = None
    if mask_kind == "padding":
        kv = rng.integers(1, N + 1, B)
    if mask_kind == "sparse":
        T = (N + 127) // 128
        bm = (rng.random((T, T)) < 0.4).astype(np.uint8)
        bm[np.arange(T), np.arange(T)] = 1
    return random_case(B, H, N, d, seed, dtype=dtype, kv_len=kv, block_mask=bm)


# every tensor in a layout other than its neighbour's, outputs included
MIXED = [
    dict(q="bnhd", k="bnhd", v="bnhd", dO="bnhd", o="bnhd", dq="bnhd", dk="bnhd", dv="bnhd"),
    dict(q="packed", k="packed", v="packed", dO="padded", o="padded", dq="hbnd", dk="packed",
         dv="bnhd"),
    dict(q="hbnd", k="padded", v="bnhd", dO="dense", o="packed", dq="padded", dk="hbnd",
         dv="padded"),
]

CASES = [
    # B, H, N, d, causal, mask
    (2, 3, 300, 64, True, "none"),
    (2, 2, 257, 128, False, "padding"),
    (1, 2, 384, 128, True, "sparse"),    # B = 1: the batch stride is ignored
    (2, 1, 200, 64, False, "none"),      # H = 1: the head stride is ignored
    (1, 1, 1, 64, False, "none"),        # one token: every stride but d's is ignored
]


@pytest.mark.parametrize("B,H,N,d,causal,mask_kind", CASES)
@pytest.mark.parametrize("mix", range(len(MIXED)))
def test_strided_bf16_equals_dense(fa, B, H, N, d, causal, mask_kind, mix):
    case = make_case(B, H, N, d, mask_kind, seed=7 * N + d + mix, dtype="bf16")
    t = to_device(case, "bf16")
    mask = fa.make_mask(t["kv_len"], t["block_mask"])
    scale = d ** -0.5
    ref = run_dense(fa, t, B, H, N, d, scale, causal, mask, fp32=False)
    got = run_strided(fa, t, (B, H, N, d), scale, causal, mask, False, MIXED[mix])
    for name, a, b in zip(("O", "lse", "dQ", "dK", "dV"), got, ref):
        assert torch.equal(a, b), name + " differs from the dense call"


@pytest.mark.parametrize("mix", range(len(MIXED)))
def test_strided_fp32_equals_dense(fa, mix):
    B, H, N, d = 2, 2, 200, 64
    case = make_case(B, H, N, d, "none", seed=31 + mix, dtype="fp32")
    t = to_device(case, "fp32")
    ref = run_dense(fa, t, B, H, N, d, 0.125, True, None, fp32=True)
    got = run_strided(fa, t, (B, H, N, d), 0.125, True, None, True, MIXED[mix])
    for name, a, b in zip(("O", "lse", "dQ", "dK", "dV"), got, ref):
        assert torch.equal(a, b), name + " differs from the dense call"


def test_strided_against_oracle(fa):
    """[B,N,H,d] inputs and outputs through the conveniences, checked against
    the fp64 oracle within the bf16 tolerances."""
    B, H, N, d = 2, 3, 333, 128
    case = make_case(B, H, N, d, "none", seed=5, dtype="bf16")
    t = to_device(case, "bf16")
    v = {n: place((B, H, N, d), torch.bfloat16, "bnhd", t[n])[1] for n in ("q", "k", "v", "do")}
    o, lse = fa.forward(v["q"], v["k"], v["v"], causal=True)
    assert o.stride() == v["q"].stride()  # O keeps the [B,N,H,d] layout
    dq, dk, dv = fa.backward(v["q"], v["k"], v["v"], o, v["do"], lse, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status()[0] == 0
    scale = d ** -0.5
    ro, rl = oracle.forward(case["q"], case["k"], case["v"], scale, causal=True)
    rdq, rdk, rdv, _ = oracle.backward(case["q"], case["k"], case["v"], case["do"], scale,
                                       causal=True)
    to, tl, tg = TOL["bf16"]
    assert max_abs(f64(o), ro) <= to
    assert max_abs(lse.cpu().numpy().astype(np.float64), rl) <= tl
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), (rdq, rdk, rdv)):
        assert rel_fro(f64(g), r) <= tg, name


def test_ignored_strides_of_size_one_dims(fa):
    """B = H = 1: batch and head strides of 0 (or anything) are ignored."""
    B, H, N, d = 1, 1, 300, 64
    case = make_case(B, H, N, d, "none", seed=11, dtype="bf16")
    t = to_device(case, "bf16")
    ref_o = torch.empty_like(t["q"])
    ref_l = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fa.fa_fwd(t["q"], t["k"], t["v"], ref_o, ref_l, B, H, N, d, 0.125, True)
    o = torch.empty_like(t["q"])
    lse = torch.empty_like(ref_l)
    ls = fa.FaLayouts()
    for name in ("q", "k", "v", "o"):
        setattr(ls, name, fa.FaLayout(0, -3, d))
    fa.fa_fwd_ex(t["q"], t["k"], t["v"], o, lse, B, H, N, d, 0.125, True, None,
                 fa.make_options(ls))
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
